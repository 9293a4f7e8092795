/*
 * mx_oracle.c -- plain, slow CPU oracle for MX-FP8 casting of bf16 matrices.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The CUDA
 * library never includes, links or calls it, and this file shares no code,
 * header, table or constant generator with the CUDA path.
 *
 * What is computed (per 32-element block, OCP Microscaling Formats (MX) v1.0,
 * conversion of a vector of scalars to an MX block, element type FP8 E4M3,
 * scale type E8M0):
 *   amax  = max |x_i| over the block
 *   e     = floor(log2(amax)) - 8        (8 = exponent of e4m3's largest
 *                                          normal, 448 = 1.75 * 2^8)
 *   e     clamped to the e8m0 range [-127, 127]; the stored byte is e + 127
 *   an all-zero block stores byte 0
 *   q_i   = e4m3(x_i * 2^-e), rounded to nearest, ties to even, and
 *           saturated to +-448 (never NaN for finite input)
 * Blocks of 32 and the two directions (dim0 = blocks along a row, dim1 =
 * blocks along a column, written out as the transposed row-major copy) follow
 * pytorch/ao PR #1869 "triton kernel to cast to mx across dim0 and dim1",
 * summary.  The per-group and per-expert variants follow pytorch/ao PR #2990
 * "[mxfp8 moe training] add compile support" (sync-free padding bound
 * rows + groups*128; 3D weights cast through a reshape to 2D).  The inverse,
 * dequantisation, takes the value of an MX element as its scale times its
 * element value (OCP MX v1.0) and rounds that product once to bf16.
 *
 * Readings taken where the pages are silent (each is repeated in the design
 * notes):
 *   - NaN or Inf anywhere in a block: scale byte 0xFF (e8m0 NaN) and every
 *     element byte 0x7F (e4m3 NaN).  No workload contains them; parity for
 *     this case is unpinned.
 *   - Blocked scale layout: the 128x4 tile layout of the 1D block-scaling
 *     factors used by NVIDIA block-scaled GEMMs (32 rows of 16 bytes per
 *     512-byte tile), zero padding to 128 rows and 4 columns.
 *
 * All floating-point work is in double, where every step here is exact: a
 * bf16 value, a product with a power of two, and the division by the e4m3
 * grid spacing are all representable.  Rounding to the e4m3 grid uses
 * nearbyint() in the default round-to-nearest-even mode.
 */
#include <fenv.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MX_BLOCK 32
#define E4M3_EMAX 8          /* largest normal e4m3 is 1.75 * 2^8 */
#define E4M3_MAXNORM 448.0
#define E8M0_BIAS 127

/* ---- scalar encodings ------------------------------------------------- */

/* Exact value of a bf16 bit pattern (1 sign, 8 exponent, 7 mantissa bits). */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int ex = (b >> 7) & 0xFF;
    int man = b & 0x7F;
    double mag;
    if (ex == 0xFF)
        return man ? NAN : (sign ? -INFINITY : INFINITY);
    if (ex == 0)
        mag = ldexp((double)man, -126 - 7);           /* subnormal */
    else
        mag = ldexp((double)(128 + man), ex - 127 - 7); /* 1.m * 2^(ex-127) */
    return sign ? -mag : mag;
}

/* e4m3fn byte nearest to v: round to nearest, ties to even, saturating at
 * +-448.  e4m3fn: bias 7, no infinities, 0x7F/0xFF are NaN, smallest normal
 * 2^-6, subnormals m * 2^-9 for m = 1..7.  The sign of zero is kept. */
uint8_t oracle_e4m3_rne_sat(double v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7E;

    /* spacing of the e4m3 grid in a's binade (3 mantissa bits) */
    double spacing;
    if (a < ldexp(1.0, -6)) {
        spacing = ldexp(1.0, -9);
    } else {
        int p;
        frexp(a, &p);                 /* a = f * 2^p, f in [0.5, 1) */
        spacing = ldexp(1.0, (p - 1) - 3);
    }
    double r = nearbyint(a / spacing) * spacing;   /* ties to even */
    if (r > E4M3_MAXNORM)
        r = E4M3_MAXNORM;                           /* saturate */

    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))                         /* subnormal */
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int p;
    double f = frexp(r, &p);                        /* r = (2f) * 2^(p-1) */
    int e = p - 1;
    int mant = (int)((2.0 * f - 1.0) * 8.0);
    return sign | (uint8_t)(((e + 7) << 3) | mant);
}

/* Element-wise oracle_e4m3_rne_sat over an array (for exhaustive checks). */
void oracle_e4m3_rne_sat_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_e4m3_rne_sat(v[i]);
}

/* e8m0 byte of one block given its elements as doubles: floor(log2 amax) - 8,
 * clamped to [-127, 127], biased by 127; zero block -> 0; NaN/Inf -> 0xFF. */
uint8_t oracle_block_scale(const double *blk, int n)
{
    double amax = 0.0;
    for (int i = 0; i < n; i++) {
        if (!isfinite(blk[i]))
            return 0xFF;
        double a = fabs(blk[i]);
        if (a > amax)
            amax = a;
    }
    if (amax == 0.0)
        return 0;
    int p;
    frexp(amax, &p);                 /* amax in [2^(p-1), 2^p) */
    int e = (p - 1) - E4M3_EMAX;
    if (e < -E8M0_BIAS)
        e = -E8M0_BIAS;
    if (e > E8M0_BIAS)
        e = E8M0_BIAS;
    return (uint8_t)(e + E8M0_BIAS);
}

/* Cast one block of n (<= 32) values with its scale byte. */
static void cast_block(const double *blk, int n, uint8_t s, uint8_t *q)
{
    for (int i = 0; i < n; i++) {
        if (s == 0xFF)
            q[i] = 0x7F;
        else
            q[i] = oracle_e4m3_rne_sat(ldexp(blk[i], E8M0_BIAS - (int)s));
    }
}

/* ---- threads ---------------------------------------------------------- */

/* Host threads that the dim0 and dim1 casts spread their rows / columns over.
 * Every row (dim0) or column (dim1) is computed by the same scalar code on its
 * own, so the result does not depend on the count; 1 (the default) runs the
 * plain sequential loops.  Built without OpenMP, the count is ignored. */
static int g_threads = 1;

void oracle_set_threads(int n)
{
    g_threads = n < 1 ? 1 : n;
}

/* Threads the casts will use (1 when built without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return g_threads;
#else
    return 1;
#endif
}

/* ---- directions ------------------------------------------------------- */

/* dim0: blocks of 32 along each row of x (M x K, row-major bf16 bits).
 * q: M x K bytes, s: M x (K/32) bytes (plain, unswizzled).  K % 32 == 0. */
void oracle_cast_dim0(const uint16_t *x, int64_t M, int64_t K, uint8_t *q, uint8_t *s)
{
    int64_t Kb = K / MX_BLOCK;
#pragma omp parallel for num_threads(g_threads) schedule(static)
    for (int64_t r = 0; r < M; r++) {
        double blk[MX_BLOCK];
        for (int64_t j = 0; j < Kb; j++) {
            for (int i = 0; i < MX_BLOCK; i++)
                blk[i] = oracle_bf16_to_double(x[r * K + j * MX_BLOCK + i]);
            uint8_t sc = oracle_block_scale(blk, MX_BLOCK);
            s[r * Kb + j] = sc;
            cast_block(blk, MX_BLOCK, sc, q + r * K + j * MX_BLOCK);
        }
    }
}

/* dim1: blocks of 32 along each column of x, written as the row-major copy of
 * the transpose: q: K x M bytes (q[k][m] encodes x[m][k]), s: K x (M/32).
 * M % 32 == 0.  Written with its own column loop (not via a transpose), so
 * that dim1(X) == dim0(X^T) is a check rather than a tautology. */
void oracle_cast_dim1(const uint16_t *x, int64_t M, int64_t K, uint8_t *q, uint8_t *s)
{
    int64_t Mb = M / MX_BLOCK;
#pragma omp parallel for num_threads(g_threads) schedule(static)
    for (int64_t k = 0; k < K; k++) {
        double blk[MX_BLOCK];
        uint8_t qb[MX_BLOCK];
        for (int64_t j = 0; j < Mb; j++) {
            for (int i = 0; i < MX_BLOCK; i++)
                blk[i] = oracle_bf16_to_double(x[(j * MX_BLOCK + i) * K + k]);
            uint8_t sc = oracle_block_scale(blk, MX_BLOCK);
            s[k * Mb + j] = sc;
            cast_block(blk, MX_BLOCK, sc, qb);
            for (int i = 0; i < MX_BLOCK; i++)
                q[k * M + j * MX_BLOCK + i] = qb[i];
        }
    }
}

/* ---- blocked (128x4) scale layout -------------------------------------- */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t oracle_blocked_bytes(int64_t R, int64_t C)
{
    return ceil_div(R, 128) * 128 * ceil_div(C, 4) * 4;
}

/* Scale matrix s (R x C, row-major) -> blocked layout of
 * ceil(R/128)*128 x ceil(C/4)*4 bytes.  Tiles of 128 rows x 4 columns are
 * stored one after another in row-major tile order, 512 bytes each; inside a
 * tile, row r and column c sit at (r % 32) * 16 + (r / 32) * 4 + c.  Padding
 * is zero. */
void oracle_to_blocked(const uint8_t *s, int64_t R, int64_t C, uint8_t *out)
{
    int64_t tiles_per_row = ceil_div(C, 4);
    memset(out, 0, (size_t)oracle_blocked_bytes(R, C));
    for (int64_t r = 0; r < R; r++) {
        for (int64_t c = 0; c < C; c++) {
            int64_t tile = (r / 128) * tiles_per_row + (c / 4);
            int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = s[r * C + c];
        }
    }
}

/* Inverse of oracle_to_blocked over the unpadded region. */
void oracle_from_blocked(const uint8_t *blk, int64_t R, int64_t C, uint8_t *s)
{
    int64_t tiles_per_row = ceil_div(C, 4);
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) {
            int64_t tile = (r / 128) * tiles_per_row + (c / 4);
            int64_t rr = r % 128, cc = c % 4;
            s[r * C + c] = blk[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc];
        }
}

/* ---- fused dim0 + dim1 with blocked scales ----------------------------- */

/* One bf16 matrix -> both copies, scales in blocked layout.  s0_blk holds
 * blk(M, K/32) bytes, s1_blk holds blk(K, M/32) bytes.  Returns 0, or -1 if
 * scratch memory could not be had. */
int oracle_cast_dim0_dim1_blocked(const uint16_t *x, int64_t M, int64_t K,
                                  uint8_t *q0, uint8_t *s0_blk,
                                  uint8_t *q1, uint8_t *s1_blk)
{
    uint8_t *s0 = malloc((size_t)(M * (K / 32)) + 1);
    uint8_t *s1 = malloc((size_t)(K * (M / 32)) + 1);
    if (!s0 || !s1) {
        free(s0);
        free(s1);
        return -1;
    }
    if (q0) {
        oracle_cast_dim0(x, M, K, q0, s0);
        oracle_to_blocked(s0, M, K / 32, s0_blk);
    }
    if (q1) {
        oracle_cast_dim1(x, M, K, q1, s1);
        oracle_to_blocked(s1, K, M / 32, s1_blk);
    }
    free(s0);
    free(s1);
    return 0;
}

/* ---- groups along M (MoE activations) ---------------------------------- */

/* Group g holds rows [o_{g-1}, o_g) with o_{-1} = 0 and offs[g] = o_g.
 *   s0_row_offs[g] = sum_{h<g} ceil(m_h/128)*128   (G+1 entries)
 *   s1_col_offs[g] = sum_{h<g} ceil(m_h/128)*4     (G+1 entries)
 * dim0: q0 and the plain scales are those of the ungrouped dim0 cast; group
 *   g's scale rows are put in blocked layout on their own and written at byte
 *   s0_row_offs[g] * ceil4(K/32) of s0_blk, which holds (M + 128 G) *
 *   ceil4(K/32) bytes, every one of them defined (padding zero).
 * dim1: group g is the dim1 cast of its own rows, zero padded to a multiple of
 *   32 rows (zeros change no block maximum and are not stored); its data goes
 *   to columns [o_{g-1}, o_g) of q1 (K x M), its scales (K x ceil(m_g/32)) in
 *   blocked layout on their own at byte ceil128(K) * s1_col_offs[g] of s1_blk,
 *   which holds ceil128(K) * (ceil(M/32) + 4 G) bytes, padding zero.
 * Empty groups (m_g = 0) take no rows and no scale space.
 * Returns 0, -1 on allocation failure, -5 on invalid offsets (decreasing,
 * negative, or last offset != M). */
int oracle_cast_grouped_m(const uint16_t *x, int64_t M, int64_t K,
                          const int32_t *offs, int G,
                          uint8_t *q0, uint8_t *s0_blk, int64_t *s0_row_offs,
                          uint8_t *q1, uint8_t *s1_blk, int64_t *s1_col_offs)
{
    if (G <= 0)
        return -5;
    int64_t prev = 0;
    for (int g = 0; g < G; g++) {
        if (offs[g] < prev || offs[g] > M)
            return -5;
        prev = offs[g];
    }
    if (prev != M)
        return -5;

    int64_t Kb = K / 32;
    int64_t Kb4 = ceil_div(Kb, 4) * 4;
    int64_t K128 = ceil_div(K, 128) * 128;
    int64_t s0_bytes = (M + 128 * (int64_t)G) * Kb4;
    int64_t s1_bytes = K128 * (ceil_div(M, 32) + 4 * (int64_t)G);

    s0_row_offs[0] = 0;
    s1_col_offs[0] = 0;
    for (int g = 0; g < G; g++) {
        int64_t lo = g ? offs[g - 1] : 0;
        int64_t mg = offs[g] - lo;
        s0_row_offs[g + 1] = s0_row_offs[g] + ceil_div(mg, 128) * 128;
        s1_col_offs[g + 1] = s1_col_offs[g] + ceil_div(mg, 128) * 4;
    }

    /* dim0 */
    uint8_t *s0 = malloc((size_t)(M * Kb) + 1);
    if (!s0)
        return -1;
    oracle_cast_dim0(x, M, K, q0, s0);
    memset(s0_blk, 0, (size_t)s0_bytes);
    for (int g = 0; g < G; g++) {
        int64_t lo = g ? offs[g - 1] : 0;
        int64_t mg = offs[g] - lo;
        if (mg == 0)
            continue;
        oracle_to_blocked(s0 + lo * Kb, mg, Kb, s0_blk + s0_row_offs[g] * Kb4);
    }
    free(s0);

    /* dim1 */
    memset(s1_blk, 0, (size_t)s1_bytes);
    for (int g = 0; g < G; g++) {
        int64_t lo = g ? offs[g - 1] : 0;
        int64_t mg = offs[g] - lo;
        if (mg == 0)
            continue;
        int64_t mp = ceil_div(mg, 32) * 32;
        uint16_t *xg = calloc((size_t)(mp * K), sizeof(uint16_t));
        uint8_t *qg = malloc((size_t)(K * mp));
        uint8_t *sg = malloc((size_t)(K * (mp / 32)));
        if (!xg || !qg || !sg) {
            free(xg);
            free(qg);
            free(sg);
            return -1;
        }
        memcpy(xg, x + lo * K, (size_t)(mg * K) * sizeof(uint16_t));
        oracle_cast_dim1(xg, mp, K, qg, sg);
        for (int64_t k = 0; k < K; k++)
            memcpy(q1 + k * M + lo, qg + k * mp, (size_t)mg);
        oracle_to_blocked(sg, K, mp / 32, s1_blk + K128 * s1_col_offs[g]);
        free(xg);
        free(qg);
        free(sg);
    }
    return 0;
}

/* ---- 3D expert weights, dim1 per expert -------------------------------- */

/* w is (E, N, K) bf16, read as the 2D matrix (E*N, K).  q1 is the dim1 copy of
 * that matrix, K x (E*N) bytes (expert e owns columns [e*N, (e+1)*N)).  Expert
 * e's scales, the (K, N/32) slice of the dim1 scale matrix, are put in blocked
 * layout on their own at byte e * blk(K, N/32).  N % 32 == 0. */
int oracle_cast_3d_dim1(const uint16_t *w, int64_t E, int64_t N, int64_t K,
                        uint8_t *q1, uint8_t *s1_blk)
{
    int64_t M = E * N;
    int64_t Mb = M / 32, Nb = N / 32;
    int64_t per = oracle_blocked_bytes(K, Nb);
    uint8_t *s1 = malloc((size_t)(K * Mb) + 1);
    uint8_t *se = malloc((size_t)(K * Nb) + 1);
    if (!s1 || !se) {
        free(s1);
        free(se);
        return -1;
    }
    oracle_cast_dim1(w, M, K, q1, s1);
    for (int64_t e = 0; e < E; e++) {
        for (int64_t k = 0; k < K; k++)
            memcpy(se + k * Nb, s1 + k * Mb + e * Nb, (size_t)Nb);
        oracle_to_blocked(se, K, Nb, s1_blk + e * per);
    }
    free(s1);
    free(se);
    return 0;
}

/* ---- 3D expert weights, dim0 per expert -------------------------------- */

/* w is (E, N, K) bf16, read as the 2D matrix (E*N, K).  q0 is its dim0 copy,
 * (E*N) x K bytes in the same order as w.  Expert e's scales are rows
 * [e*N, (e+1)*N) of the dim0 scale matrix, an (N, K/32) block that is put in
 * blocked layout on its own at byte e * blk(N, K/32).  K % 32 == 0; N >= 1
 * need not be a multiple of 32 (dim0 blocks run along K). */
int oracle_cast_3d_dim0(const uint16_t *w, int64_t E, int64_t N, int64_t K,
                        uint8_t *q0, uint8_t *s0_blk)
{
    int64_t M = E * N, Kb = K / 32;
    int64_t per = oracle_blocked_bytes(N, Kb);
    uint8_t *s0 = malloc((size_t)(M * Kb) + 1);
    if (!s0)
        return -1;
    oracle_cast_dim0(w, M, K, q0, s0);
    for (int64_t e = 0; e < E; e++)
        oracle_to_blocked(s0 + e * N * Kb, N, Kb, s0_blk + e * per);
    free(s0);
    return 0;
}

/* ---- dequantisation --------------------------------------------------- */

/* Exact value of an e4m3fn byte (NaN for 0x7F / 0xFF). */
double oracle_e4m3_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int ex = (b >> 3) & 0xF;
    int man = b & 0x7;
    double mag;
    if (ex == 0xF && man == 0x7)
        return NAN;
    if (ex == 0)
        mag = ldexp((double)man, -9);
    else
        mag = ldexp((double)(8 + man), ex - 7 - 3);
    return sign ? -mag : mag;
}

/* bf16 bit pattern nearest to v: round to nearest, ties to even, over the
 * whole bf16 range (subnormals m * 2^-133 kept; a magnitude that rounds to
 * 2^128 or beyond becomes infinity, as in IEEE 754 rounding).  NaN -> 0x7FC0. */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int p;
    frexp(a, &p);                       /* a in [2^(p-1), 2^p) */
    int e = p - 1;
    if (e < -126)
        e = -126;                       /* subnormal range: fixed spacing 2^-133 */
    double spacing = ldexp(1.0, e - 7); /* 7 fraction bits */
    double r = nearbyint(a / spacing) * spacing;
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    if (r < ldexp(1.0, -126))           /* subnormal (or zero) */
        return sign | (uint16_t)(r / ldexp(1.0, -133));
    double f = frexp(r, &p);            /* r = (2f) * 2^(p-1) */
    int ex = p - 1;
    int mant = (int)((2.0 * f - 1.0) * 128.0);
    return sign | (uint16_t)(((ex + 127) << 7) | mant);
}

/* MX dequantisation of one matrix: q (R x C e4m3 bytes, blocks of 32 along
 * rows, C % 32 == 0) and its scales in blocked layout (blk(R, C/32) bytes) ->
 * bf16 bits out[r][c] = bf16(e4m3(q[r][c]) * 2^(s - 127)), where s is the
 * scale byte of (r, c / 32).  The value of an MX element is the product of
 * its scale and its element value (OCP MX v1.0); the product is exact in
 * double and rounded once to bf16.  A NaN scale (0xFF) or NaN element gives
 * NaN (0x7FC0).  Returns 0, or -1 if scratch memory could not be had. */
int oracle_dequant_blocked(const uint8_t *q, int64_t R, int64_t C, const uint8_t *s_blk,
                           uint16_t *out)
{
    int64_t Cb = C / MX_BLOCK;
    uint8_t *s = malloc((size_t)(R * Cb) + 1);
    if (!s)
        return -1;
    oracle_from_blocked(s_blk, R, Cb, s);
    for (int64_t r = 0; r < R; r++) {
        for (int64_t c = 0; c < C; c++) {
            uint8_t sc = s[r * Cb + c / MX_BLOCK];
            double v = oracle_e4m3_to_double(q[r * C + c]);
            if (sc == 0xFF || isnan(v))
                out[r * C + c] = 0x7FC0;
            else
                out[r * C + c] = oracle_double_to_bf16(ldexp(v, (int)sc - E8M0_BIAS));
        }
    }
    free(s);
    return 0;
}

/* ---- tensorwise and rowwise fp8 (non-MX contrast cases) ----------------- */

/* Nearest fp32 to v (the C conversion double -> float rounds to nearest even). */
static double to_f32(double v)
{
    return (double)(float)v;
}

/* Tensorwise fp8 with one dynamic scale for the whole tensor, as in pytorch/ao
 * PR #1445 "[float8nocompile] Triton kernels for conversion to float8 dtypes"
 * (global amax over all elements, then one scale, then the conversion):
 *   amax  = max |x_i|                                   (exact)
 *   scale = fp32 nearest to 448 / amax; amax = 0 gives 1; a quotient beyond
 *           the largest finite fp32 gives the largest finite fp32
 *   q_i   = e4m3(fp32(x_i * scale)), nearest even, saturated to +-448
 * x holds n bf16 bit patterns; q gets n bytes.  NaN / Inf inputs follow IEEE
 * arithmetic through the same formula. */
void oracle_cast_tensorwise(const uint16_t *x, int64_t n, uint8_t *q, float *scale,
                            float *amax_out)
{
    double amax = 0.0;
    int nan = 0;
    for (int64_t i = 0; i < n; i++) {
        double v = oracle_bf16_to_double(x[i]);
        if (isnan(v))
            nan = 1;
        else if (fabs(v) > amax)
            amax = fabs(v);
    }
    if (nan)
        amax = NAN;
    double s;
    if (amax == 0.0)
        s = 1.0;
    else {
        s = to_f32(E4M3_MAXNORM / amax);
        if (isinf(s))
            s = (double)FLT_MAX;
    }
    for (int64_t i = 0; i < n; i++)
        q[i] = oracle_e4m3_rne_sat(to_f32(oracle_bf16_to_double(x[i]) * s));
    *scale = (float)s;
    *amax_out = (float)amax;
}

/* Rowwise fp8 with one scale per row, as in the "FP8 linear triton with
 * row-wise scaling" gist (quantize_fp8_rowwise):
 *   amax_r  = max_j |x_rj|                               (exact)
 *   scale_r = bf16 nearest to amax_r / 448 (the input's dtype)
 *   q_rj    = e4m3(fp32(x_rj / scale_r)), nearest even, saturated to +-448
 * A row whose scale is 0 (all zero, or amax_r / 448 below half the smallest
 * bf16 subnormal) encodes as signed zeros instead of the formula's 0/0.
 * x is M x K bf16 bits; q gets M x K bytes, scale M bf16 bit patterns. */
void oracle_cast_rowwise(const uint16_t *x, int64_t M, int64_t K, uint8_t *q, uint16_t *scale)
{
    for (int64_t r = 0; r < M; r++) {
        const uint16_t *xr = x + r * K;
        double amax = 0.0;
        int nan = 0;
        for (int64_t j = 0; j < K; j++) {
            double v = oracle_bf16_to_double(xr[j]);
            if (isnan(v))
                nan = 1;
            else if (fabs(v) > amax)
                amax = fabs(v);
        }
        if (nan)
            amax = NAN;
        uint16_t sb = oracle_double_to_bf16(amax / E4M3_MAXNORM);
        double s = oracle_bf16_to_double(sb);
        scale[r] = sb;
        for (int64_t j = 0; j < K; j++) {
            double v = oracle_bf16_to_double(xr[j]);
            if (s == 0.0)
                q[r * K + j] = signbit(v) ? 0x80 : 0x00;
            else
                q[r * K + j] = oracle_e4m3_rne_sat(to_f32(v / s));
        }
    }
}
