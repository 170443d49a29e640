/*
 * bsf8_oracle.c -- plain, slow CPU oracle for the block-scaled FP8 weight path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and its
 * reference arm) load it.  It shares no code, header, table or helper with the
 * CUDA library; its number codecs are written here from the format definitions.
 *
 * Sources (titles of the pages this restates; section names in brackets):
 *   [twin]  "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" -- module docstring,
 *           make_twin(), _wo_a_partial_w8(), _wo_a_mid_kernel(), _dequant_kernel().
 *   [pad]   "recipes/docker-images/mia-tp4/adapter/shared_pad_k.py" -- docstring
 *           sections LOSSLESS and WHAT THE PATCH DOES, _pad_weight(), _pad_input().
 *
 * Number formats (OCP 8-bit floating point, E4M3 "fn" variant; bfloat16):
 *   e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
 *         holds subnormals m*2^-9; no infinities; S.1111.111 is NaN; largest finite
 *         magnitude 448.
 *   bf16: the upper 16 bits of an IEEE binary32; conversion from binary32 rounds to
 *         nearest, ties to even.
 *
 * Every floating-point step is an explicit binary32 (or, where named, binary64)
 * operation.  Build with -O1 -ffp-contract=off -fno-fast-math so that no multiply
 * and add are fused and no operation is reassociated.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py against
 * library casts (torch), closed forms derived by hand (tests/golden/), integer
 * arithmetic, binary64 sums with Higham's bound, and the pages' printed facts.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stddef.h>

/* ------------------------------------------------------------------ bf16 */

float bsfo_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even.  Adding 0x7FFF plus the lowest
 * kept bit to the full pattern and truncating rounds the dropped 16 bits correctly in
 * every binade, including the subnormal range and the carry into infinity.  NaN keeps
 * its sign and becomes a quiet NaN. */
uint16_t bsfo_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + keep_lsb) >> 16);
}

/* ------------------------------------------------------------------ e4m3 */

float bsfo_e4m3_decode(uint8_t b)
{
    int sign = b >> 7;
    int ef = (b >> 3) & 0xF;
    int m = b & 7;
    float v;
    if (ef == 15 && m == 7)
        return sign ? -NAN : NAN;
    if (ef == 0)
        v = ldexpf((float)m, -9);               /* m/8 * 2^-6 */
    else
        v = ldexpf((float)(8 + m), ef - 7 - 3); /* (1 + m/8) * 2^(ef-7) */
    return sign ? -v : v;
}

/* binary32 -> e4m3, round to nearest, ties to even.  The quantum of the binade that
 * holds |x| is 2^(floor(log2|x|) - 3), never finer than the subnormal quantum 2^-9;
 * |x| / quantum is rounded with rint (round-half-even in the default mode) and the
 * rounded magnitude is re-encoded.  A result above 448 has no e4m3 encoding and maps
 * to NaN (the "fn" variant has no infinity); NaN input maps to NaN. */
uint8_t bsfo_e4m3_rne(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    float a = fabsf(x);
    if (isinf(a))
        return (uint8_t)(sign | 0x7F);
    if (a == 0.0f)
        return sign;
    int ex;
    (void)frexpf(a, &ex);           /* a = fr * 2^ex, fr in [0.5, 1): floor(log2 a) = ex-1 */
    int e_unb = ex - 1;
    if (e_unb < -6)
        e_unb = -6;                 /* subnormal binade shares the 2^-9 quantum */
    float quantum = ldexpf(1.0f, e_unb - 3);
    float r = rintf(a / quantum);   /* exact division by a power of two, then RNE */
    float v = r * quantum;          /* exact */
    if (v == 0.0f)
        return sign;
    if (v > 448.0f)
        return (uint8_t)(sign | 0x7F);
    (void)frexpf(v, &ex);
    int ev = ex - 1;
    if (ev < -6) {                  /* subnormal: v = m * 2^-9, m in 1..7 */
        int m = (int)ldexpf(v, 9);
        return (uint8_t)(sign | m);
    }
    int m = (int)ldexpf(v, 3 - ev) - 8;   /* v = (8+m) * 2^(ev-3) */
    return (uint8_t)(sign | ((ev + 7) << 3) | m);
}

/* -------------------------------------------------------------- dequant */

/* [twin] _dequant_kernel / the in-register rebuild in _wo_a_partial_w8:
 *   W = bf16( float(q) * 2^(e_byte - 127) ).
 * The pages write the scale as exp2(e - 127.0); for an integer argument that is the
 * power of two ldexpf(1, e-127) (2^-127 is a binary32 subnormal, 2^128 is +inf). */
uint16_t bsfo_dequant_one(uint8_t q, uint8_t e_byte)
{
    float scale = ldexpf(1.0f, (int)e_byte - 127);
    float p = bsfo_e4m3_decode(q) * scale;
    return bsfo_bf16_rne(p);
}

/* w8[G][N][K] codes, ex[G][N/32][K/32] exponent bytes -> out[G][N][K] bf16 bits. */
void bsfo_dequant(const uint8_t *w8, const uint8_t *ex, uint16_t *out, int G, int N, int K)
{
    int nb = N / 32, kb = K / 32;
    for (int g = 0; g < G; ++g)
        for (int n = 0; n < N; ++n)
            for (int k = 0; k < K; ++k) {
                size_t i = ((size_t)g * N + n) * K + k;
                uint8_t e = ex[((size_t)g * nb + n / 32) * kb + k / 32];
                out[i] = bsfo_dequant_one(w8[i], e);
            }
}

/* ------------------------------------------------------------ make_twin */

/* [twin] make_twin(): the block exponent for a finite block maximum |w| = amax:
 * amax is raised to at least 2^-126, then e = ceil(log2(amax / 448)) clamped to
 * [-127, 127]. */
int bsfo_twin_exponent(float amax)
{
    const float floor_amax = ldexpf(1.0f, -126);
    if (amax < floor_amax)
        amax = floor_amax;
    double t = ceil(log2((double)amax / 448.0));
    if (t < -127.0)
        t = -127.0;
    if (t > 127.0)
        t = 127.0;
    return (int)t;
}

/* [twin] make_twin(), per 32x32 block of a bf16 weight:
 *   amax  = max |w| over the block, raised to at least 2^-126;
 *   e     = ceil(log2(amax / 448)), clamped to [-127, 127];
 *   q     = e4m3(w / 2^e)                     (binary32 divide, RNE cast);
 *   back  = bf16(float(q) * 2^e)              (binary32 multiply, RNE cast);
 *   the twin is kept only if back == w for every element of the tensor
 *   (value equality, so -0 == +0);  exponent byte = e + 127.
 * The pages leave blocks holding NaN or Inf undefined; this oracle (and the library)
 * marks them: block flag 0, exponent byte 0xFF, every code 0x7F.  Such a tensor is
 * rejected either way, as it is on the pages.
 * The log2 is taken in binary64; for every bf16 amax the result equals the binary32
 * expression on the pages (pinned by brute force over all bf16 patterns).
 * Returns 1 if the whole tensor reproduces, else 0.  ok[] may be NULL. */
int bsfo_make_twin(const uint16_t *w, uint8_t *w8, uint8_t *ex, uint8_t *ok,
                   int G, int N, int K)
{
    int nb = N / 32, kb = K / 32;
    int accepted = 1;
    for (int g = 0; g < G; ++g)
        for (int bi = 0; bi < nb; ++bi)
            for (int bj = 0; bj < kb; ++bj) {
                size_t blk = ((size_t)g * nb + bi) * kb + bj;
                float amax = 0.0f;
                int nonfinite = 0;
                for (int r = 0; r < 32; ++r)
                    for (int c = 0; c < 32; ++c) {
                        size_t i = ((size_t)g * N + bi * 32 + r) * K + bj * 32 + c;
                        float a = fabsf(bsfo_bf16_to_f32(w[i]));
                        if (!isfinite(a))
                            nonfinite = 1;
                        else if (a > amax)
                            amax = a;
                    }
                if (nonfinite) {
                    for (int r = 0; r < 32; ++r)
                        for (int c = 0; c < 32; ++c)
                            w8[((size_t)g * N + bi * 32 + r) * K + bj * 32 + c] = 0x7F;
                    ex[blk] = 0xFF;
                    if (ok)
                        ok[blk] = 0;
                    accepted = 0;
                    continue;
                }
                int e = bsfo_twin_exponent(amax);
                float scale = ldexpf(1.0f, e);
                int block_ok = 1;
                for (int r = 0; r < 32; ++r)
                    for (int c = 0; c < 32; ++c) {
                        size_t i = ((size_t)g * N + bi * 32 + r) * K + bj * 32 + c;
                        float wf = bsfo_bf16_to_f32(w[i]);
                        uint8_t q = bsfo_e4m3_rne(wf / scale);
                        float back = bsfo_bf16_to_f32(bsfo_bf16_rne(bsfo_e4m3_decode(q) * scale));
                        w8[i] = q;
                        if (!(back == wf))
                            block_ok = 0;
                    }
                ex[blk] = (uint8_t)(e + 127);
                if (ok)
                    ok[blk] = (uint8_t)block_ok;
                if (!block_ok)
                    accepted = 0;
            }
    return accepted;
}

/* ----------------------------------------------------------------- GEMM */

/* [twin] the grouped small-M linear (einsum "bgd,grd->bgr" in the draft, and the
 * partial kernels' tile loop):
 *   y[m][g][n] = bf16( sum_{k=0..K-1} float(x[m][g*K + k]) * float(W[g][n][k]) )
 * with W the exact bf16 dequant above, x[m] a row of stride ldx (>= G*K) bf16
 * elements, and the sum a binary32 running sum taken in increasing k, starting from
 * +0.  Product and sum are separate binary32 operations. */
void bsfo_gemm(const uint16_t *x, long ldx, const uint8_t *w8, const uint8_t *ex,
               uint16_t *y, int M, int N, int K, int G)
{
    int nb = N / 32, kb = K / 32;
    (void)nb;
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g)
            for (int n = 0; n < N; ++n) {
                float acc = 0.0f;
                const uint8_t *wrow = w8 + ((size_t)g * N + n) * K;
                const uint8_t *erow = ex + ((size_t)g * (N / 32) + n / 32) * kb;
                const uint16_t *xrow = x + (size_t)m * ldx + (size_t)g * K;
                for (int k = 0; k < K; ++k) {
                    float wv = bsfo_bf16_to_f32(bsfo_dequant_one(wrow[k], erow[k / 32]));
                    float xv = bsfo_bf16_to_f32(xrow[k]);
                    float p = xv * wv;
                    acc = acc + p;
                }
                y[((size_t)m * G + g) * N + n] = bsfo_bf16_rne(acc);
            }
}

/* Same sum in binary64 (each product is exact in binary64), unrounded; used to check
 * the binary32 oracle against Higham's bound.  Also returns sum |x*w| in absprod. */
void bsfo_gemm_f64(const uint16_t *x, long ldx, const uint8_t *w8, const uint8_t *ex,
                   double *y, double *absprod, int M, int N, int K, int G)
{
    int kb = K / 32;
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g)
            for (int n = 0; n < N; ++n) {
                double acc = 0.0, aacc = 0.0;
                const uint8_t *wrow = w8 + ((size_t)g * N + n) * K;
                const uint8_t *erow = ex + ((size_t)g * (N / 32) + n / 32) * kb;
                const uint16_t *xrow = x + (size_t)m * ldx + (size_t)g * K;
                for (int k = 0; k < K; ++k) {
                    double wv = bsfo_bf16_to_f32(bsfo_dequant_one(wrow[k], erow[k / 32]));
                    double xv = bsfo_bf16_to_f32(xrow[k]);
                    acc += xv * wv;
                    aacc += fabs(xv * wv);
                }
                y[((size_t)m * G + g) * N + n] = acc;
                absprod[((size_t)m * G + g) * N + n] = aacc;
            }
}

/* ------------------------------------------------------------- split-K */

/* Split s of S covers whole 32-column blocks: chunk = ceil((K/32)/S) blocks, split s
 * spans columns [s*chunk*32, min(K, (s+1)*chunk*32)) and may be empty.  (The pages
 * split K=4096 into equal parts; this is the same rule where S divides K/32.) */
void bsfo_split_range(int K, int S, int s, int *k_lo, int *k_hi)
{
    int nkb = K / 32;
    int chunk = (nkb + S - 1) / S;
    int lo = s * chunk * 32, hi = (s + 1) * chunk * 32;
    if (lo > K) lo = K;
    if (hi > K) hi = K;
    *k_lo = lo;
    *k_hi = hi;
}

/* [twin] _wo_a_partial_w8 / _wo_a_mid_kernel with SPLIT_K > 1: split s writes the
 * binary32 partial P[s][m][g][n] of its column range (running sum in increasing k,
 * from +0). */
void bsfo_gemm_partials(const uint16_t *x, long ldx, const uint8_t *w8, const uint8_t *ex,
                        float *P, int M, int N, int K, int G, int S)
{
    int kb = K / 32;
    for (int s = 0; s < S; ++s) {
        int lo, hi;
        bsfo_split_range(K, S, s, &lo, &hi);
        for (int m = 0; m < M; ++m)
            for (int g = 0; g < G; ++g)
                for (int n = 0; n < N; ++n) {
                    float acc = 0.0f;
                    const uint8_t *wrow = w8 + ((size_t)g * N + n) * K;
                    const uint8_t *erow = ex + ((size_t)g * (N / 32) + n / 32) * kb;
                    const uint16_t *xrow = x + (size_t)m * ldx + (size_t)g * K;
                    for (int k = lo; k < hi; ++k) {
                        float wv = bsfo_bf16_to_f32(bsfo_dequant_one(wrow[k], erow[k / 32]));
                        float xv = bsfo_bf16_to_f32(xrow[k]);
                        float p = xv * wv;
                        acc = acc + p;
                    }
                    P[(((size_t)s * M + m) * G + g) * N + n] = acc;
                }
    }
}

/* [twin] the fixed-order second pass (partial.sum(0) / reduce_k): for every output
 *   y = bf16( ((P[0] + P[1]) + P[2]) + ... + P[S-1] ),
 * summed left to right in binary32, one rounding to bf16 at the end. */
void bsfo_splitk_reduce(const float *P, uint16_t *y, long count, int S)
{
    for (long i = 0; i < count; ++i) {
        float acc = P[i];
        for (int s = 1; s < S; ++s)
            acc = acc + P[(size_t)s * count + i];
        y[i] = bsfo_bf16_rne(acc);
    }
}

/* ---------------------------------------------------------------- pad-K */

/* [pad] _pad_weight(): the weight [N][K] becomes [N][Kp] with zero weights in the new
 * columns and its 32x32 scales [N/32][K/32] become [N/32][Kp/32] with scale 1.0
 * (exponent byte 127 by default; the pages checked that 0, 127 and 200 give the same
 * output).  Applied to every group g of a [G][N][K] weight. */
void bsfo_pad_k(const uint8_t *w8, const uint8_t *ex, uint8_t *w8_out, uint8_t *ex_out,
                int G, int N, int K, int Kp, uint8_t pad_exp)
{
    int nb = N / 32, kb = K / 32, kbp = Kp / 32;
    for (int g = 0; g < G; ++g)
        for (int n = 0; n < N; ++n)
            for (int k = 0; k < Kp; ++k)
                w8_out[((size_t)g * N + n) * Kp + k] =
                    k < K ? w8[((size_t)g * N + n) * K + k] : (uint8_t)0x00;
    for (int g = 0; g < G; ++g)
        for (int b = 0; b < nb; ++b)
            for (int j = 0; j < kbp; ++j)
                ex_out[((size_t)g * nb + b) * kbp + j] =
                    j < kb ? ex[((size_t)g * nb + b) * kb + j] : pad_exp;
}

/* [pad] _pad_input(): the activation row [G*K] (stride ldx) becomes [G*Kp] with +0 in
 * every new column. */
void bsfo_pad_x(const uint16_t *x, long ldx, uint16_t *x_out, int M, int G, int K, int Kp)
{
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g)
            for (int k = 0; k < Kp; ++k)
                x_out[(size_t)m * G * Kp + (size_t)g * Kp + k] =
                    k < K ? x[(size_t)m * ldx + (size_t)g * K + k] : (uint16_t)0x0000;
}

/* ------------------------------------------- per-(row, 32-column) scales */

/* The pages' second twin layout ("recipes/docker-images/mia-tp4/docs/tp4-adapters.md",
 * adapter table, draft_main_proj): e4m3 codes with one power-of-two scale per (weight
 * row, 32 columns), checked to reproduce the bf16 weight exactly.  The pages give no
 * formula for it; this oracle takes make_twin's rule with the block narrowed to 1 x 32:
 * the exponent layout is ex[G][N][K/32], everything else as above. */

/* w8[G][N][K] codes, ex[G][N][K/32] exponent bytes -> out[G][N][K] bf16 bits. */
void bsfo_dequant_rows(const uint8_t *w8, const uint8_t *ex, uint16_t *out, int G, int N, int K)
{
    int kb = K / 32;
    for (int g = 0; g < G; ++g)
        for (int n = 0; n < N; ++n)
            for (int k = 0; k < K; ++k) {
                size_t i = ((size_t)g * N + n) * K + k;
                uint8_t e = ex[((size_t)g * N + n) * kb + k / 32];
                out[i] = bsfo_dequant_one(w8[i], e);
            }
}

/* make_twin with 1 x 32 blocks: per (row n, columns 32j .. 32j+31), amax over those 32
 * values, the same exponent rule, codes and exact-rebuild check, and the same marking of
 * blocks that hold NaN or Inf.  ex, ok: [G][N][K/32].  Returns 1 if every element
 * reproduces. */
int bsfo_make_twin_rows(const uint16_t *w, uint8_t *w8, uint8_t *ex, uint8_t *ok,
                        int G, int N, int K)
{
    int kb = K / 32;
    int accepted = 1;
    for (int g = 0; g < G; ++g)
        for (int n = 0; n < N; ++n)
            for (int bj = 0; bj < kb; ++bj) {
                size_t blk = ((size_t)g * N + n) * kb + bj;
                size_t base = ((size_t)g * N + n) * K + (size_t)bj * 32;
                float amax = 0.0f;
                int nonfinite = 0;
                for (int c = 0; c < 32; ++c) {
                    float a = fabsf(bsfo_bf16_to_f32(w[base + c]));
                    if (!isfinite(a))
                        nonfinite = 1;
                    else if (a > amax)
                        amax = a;
                }
                if (nonfinite) {
                    for (int c = 0; c < 32; ++c)
                        w8[base + c] = 0x7F;
                    ex[blk] = 0xFF;
                    if (ok)
                        ok[blk] = 0;
                    accepted = 0;
                    continue;
                }
                int e = bsfo_twin_exponent(amax);
                float scale = ldexpf(1.0f, e);
                int block_ok = 1;
                for (int c = 0; c < 32; ++c) {
                    float wf = bsfo_bf16_to_f32(w[base + c]);
                    uint8_t q = bsfo_e4m3_rne(wf / scale);
                    float back = bsfo_bf16_to_f32(bsfo_bf16_rne(bsfo_e4m3_decode(q) * scale));
                    w8[base + c] = q;
                    if (!(back == wf))
                        block_ok = 0;
                }
                ex[blk] = (uint8_t)(e + 127);
                if (ok)
                    ok[blk] = (uint8_t)block_ok;
                if (!block_ok)
                    accepted = 0;
            }
    return accepted;
}

/* The GEMM of bsfo_gemm with the weight rebuilt from per-(row, 32-column) exponents. */
void bsfo_gemm_rows(const uint16_t *x, long ldx, const uint8_t *w8, const uint8_t *ex,
                    uint16_t *y, int M, int N, int K, int G)
{
    int kb = K / 32;
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g)
            for (int n = 0; n < N; ++n) {
                float acc = 0.0f;
                const uint8_t *wrow = w8 + ((size_t)g * N + n) * K;
                const uint8_t *erow = ex + ((size_t)g * N + n) * kb;
                const uint16_t *xrow = x + (size_t)m * ldx + (size_t)g * K;
                for (int k = 0; k < K; ++k) {
                    float wv = bsfo_bf16_to_f32(bsfo_dequant_one(wrow[k], erow[k / 32]));
                    float xv = bsfo_bf16_to_f32(xrow[k]);
                    float p = xv * wv;
                    acc = acc + p;
                }
                y[((size_t)m * G + g) * N + n] = bsfo_bf16_rne(acc);
            }
}

/* ------------------------------------------------------- array wrappers */

/* Element-wise loops over the scalar codecs above, so tests can sweep millions of
 * values without one foreign call per value. */
void bsfo_bf16_rne_array(const float *in, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bsfo_bf16_rne(in[i]);
}

void bsfo_e4m3_rne_array(const float *in, uint8_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bsfo_e4m3_rne(in[i]);
}

void bsfo_e4m3_decode_array(const uint8_t *in, float *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bsfo_e4m3_decode(in[i]);
}

void bsfo_twin_exponent_array(const float *amax, int *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = bsfo_twin_exponent(amax[i]);
}
