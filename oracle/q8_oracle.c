/*
 * Q8_0 oracle: a plain, slow, obviously correct CPU statement of the Q8_0
 * row quantizer and of the qdot_t contraction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library (gemm_q8_qdot_gb300/csrc),
 * and the product path never calls it.
 *
 * Sources (Phobos documentation pages):
 *   - "Quantized built-ins and formats" (phobos-lang.dev/docs/language/quantized/),
 *     section "Q8_0": the block format (signed bytes, one scale per block of 32,
 *     activations quantized the same way) and the qdot_t formula
 *       out[i,j] = sum_b a_scales[i,b] * w_scales[j,b] * sum_{k in b} a[i,k] * w[j,k]
 *     with the inner sum in integers.
 *   - "Phobos Language Spec" (phobos-lang.dev/docs/reference/spec/), section 10
 *     "Quantized built-ins", Q8_0 table: shapes a [M,K] i8, w [N,K] i8, scales
 *     [M,K/32] and [N,K/32] f32, out [M,N] f32; qmma_t takes w_scales as
 *     [K/32, N].
 *   - Same spec, section 9 "Built-ins", Elementwise table: round() is the
 *     nearest integer with ties to even.
 *   - Same spec, section 3 "Types": i8 loads sign-extend.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *   - The scale of a block is d = amax / 127 in f32, amax = max |x| over the
 *     block, q = round_ties_even(x / d) clamped to [-127, 127]; a block with
 *     d == 0 stores q = 0.  (The pages only say activations are "quantized the
 *     same way"; this is the plainest reading that fits a signed-byte format
 *     with a per-block f32 scale.)
 *   - x / d is one IEEE f32 division; round() is ties-to-even.
 *
 * Precision: the quantizer runs in f32 (its outputs are f32 scales and bytes,
 * fixed bit for bit by the reading above).  Block sums run in int64 (exact).
 * The scaled sum runs in double; `bound` returns 1e-5 * sum_b |t_b| + 1e-6,
 * t_b = a_scales[i,b] * w_scales[j,b] * S[i,j,b], the tolerance an f32
 * implementation is held to.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no contraction of a*b+c into an FMA, no fast math: the quantizer's bytes
 * must be the IEEE ones).
 *
 * ORACLE_MUTANT (compile-time, test only): when defined to a non-zero value
 * the library is built with one deliberate, plausible mistake, so that a test
 * can show the pins catch it.  The default build defines nothing.
 *
 * Threads: built with -fopenmp, the loops over quantizer rows and over output
 * elements (i, j) are shared among the host cores.  Each row and each output
 * element is still computed by the same sequential loop as in the
 * single-thread build, so both builds give the same bytes; without -fopenmp
 * the pragmas are ignored.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <fenv.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define QK 32 /* elements per Q8_0 block */

int oracle_mutant(void) { return ORACLE_MUTANT; }

/* Threads the parallel loops use: 1 in the single-thread build. */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* round(t): nearest integer, ties to even (spec section 9, Elementwise). */
static float round_ties_even(float v) {
#if ORACLE_MUTANT == 1
    return roundf(v); /* mutant: ties away from zero */
#elif ORACLE_MUTANT == 2
    return truncf(v); /* mutant: truncation, the float->int conversion rule */
#else
    return nearbyintf(v); /* default rounding mode is to nearest, ties to even */
#endif
}

/*
 * Row quantizer f32 -> Q8_0.  x [rows, K] f32, q [rows, K] i8, s [rows, K/32] f32.
 * Per row r and block b: amax = max |x|, d = amax / 127, q = clamp(round(x / d)).
 */
void oracle_quantize_q8_0(const float* x, int8_t* q, float* s, int64_t rows, int64_t K) {
    const int64_t KB = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        fesetround(FE_TONEAREST); /* per thread: the rounding mode is thread-local */
        for (int64_t b = 0; b < KB; ++b) {
            const float* xb = x + r * K + b * QK;
            int8_t* qb = q + r * K + b * QK;
            float amax = 0.0f;
            for (int k = 0; k < QK; ++k) {
                float v = fabsf(xb[k]);
                if (v > amax) amax = v;
            }
#if ORACLE_MUTANT == 3
            float d = amax / 128.0f; /* mutant: wrong divisor */
#else
            float d = amax / 127.0f;
#endif
            s[r * KB + b] = d;
            for (int k = 0; k < QK; ++k) {
                if (d == 0.0f) {
                    qb[k] = 0;
                    continue;
                }
                float v = round_ties_even(xb[k] / d);
                if (v > 127.0f) v = 127.0f;
                if (v < -127.0f) v = -127.0f;
                qb[k] = (int8_t)v;
            }
        }
    }
}

/*
 * Integer block sums S[i, j, b] = sum_{k in block b} a[i,k] * w[j,k], exact in
 * int64.  a [M, K] i8, w [N, K] i8 (both row-major, K contiguous), S [M, N, K/32].
 */
void oracle_blocksums_q8_0(const int8_t* a, const int8_t* w, int64_t* S,
                           int64_t M, int64_t N, int64_t K) {
    const int64_t KB = K / QK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            for (int64_t b = 0; b < KB; ++b) {
                int64_t acc = 0;
                for (int64_t k = b * QK; k < (b + 1) * QK; ++k) {
#if ORACLE_MUTANT == 5
                    acc += (int64_t)(uint8_t)a[i * K + k] * (int64_t)w[j * K + k]; /* mutant: zero-extended a */
#else
                    acc += (int64_t)a[i * K + k] * (int64_t)w[j * K + k];
#endif
                }
                S[(i * N + j) * KB + b] = acc;
            }
}

/*
 * qdot_t: out[i, j] = sum_b as[i, b] * ws(j, b) * S[i, j, b] in double, plus the
 * tolerance bound[i, j] = 1e-5 * sum_b |t_b| + 1e-6.
 * a [M,K] i8, as [M,K/32] f32, w [N,K] i8, ws f32, out / bound [M,N] f64.
 * ws_layout 0: ws is [N, K/32] (qdot_t); 1: ws is [K/32, N] (qmma_t).
 */
void oracle_qdot_q8_0_ex(const int8_t* a, const float* as, const int8_t* w, const float* ws,
                         double* out, double* bound, int64_t M, int64_t N, int64_t K,
                         int ws_layout) {
    const int64_t KB = K / QK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double T = 0.0, U = 0.0;
#if ORACLE_MUTANT == 6
            for (int64_t b = 0; b + 1 < KB; ++b) { /* mutant: last block dropped */
#else
            for (int64_t b = 0; b < KB; ++b) {
#endif
                int64_t S = 0;
                for (int64_t k = b * QK; k < (b + 1) * QK; ++k)
                    S += (int64_t)a[i * K + k] * (int64_t)w[j * K + k];
                double wsb = ws_layout ? (double)ws[b * N + j] : (double)ws[j * KB + b];
#if ORACLE_MUTANT == 7
                double asb = (double)as[b]; /* mutant: activation scale row ignored */
#else
                double asb = (double)as[i * KB + b];
#endif
                double t = asb * wsb * (double)S;
                T += t;
                U += fabs(t);
            }
            out[i * N + j] = T;
            if (bound) bound[i * N + j] = 1e-5 * U + 1e-6;
        }
}

void oracle_qdot_q8_0(const int8_t* a, const float* as, const int8_t* w, const float* ws,
                      double* out, double* bound, int64_t M, int64_t N, int64_t K) {
#if ORACLE_MUTANT == 8
    /* mutant: weight row index transposed with the activation row index */
    oracle_qdot_q8_0_ex(w, ws, a, as, out, bound, N, M, K, 0);
    (void)0;
#else
    oracle_qdot_q8_0_ex(a, as, w, ws, out, bound, M, N, K, 0);
#endif
}

/* ------------------------------------------------------------------ Q5_0 weights
 *
 * q50_qdot_t ("Phobos Language Spec" section 10, Q5_0 row; "Quantized built-ins
 * and formats", built-in table): qdot_t against a Q5_0 weight held as its
 * blocks without their f16 scale.  Per 32 elements a block is 20 bytes: the qh
 * word, then 16 bytes whose byte e holds element e in its low nibble and
 * element e + 16 in its high nibble; each element is q - 16, widened as it is
 * loaded; the scales are as for qdot_t (w_scales [N, K/32] f32, or [K/32, N]
 * for q50_qmma_t).
 *
 * Reading (the pages do not spell out the qh bit order): qh is a little-endian
 * 32-bit word and its bit e is the fifth bit (value 16) of element e, so
 * q = nibble(e) | (((qh >> e) & 1) << 4).
 *
 * w5 [N, K/32 * 20] bytes, row-major, block b of row j at byte j*(K/32)*20 + 20*b.
 */
#define Q50_BYTES 20

static int q50_value(const uint8_t* blk, int e) {
    const uint32_t qh = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8) | ((uint32_t)blk[2] << 16) |
                        ((uint32_t)blk[3] << 24);
    const uint8_t byte = blk[4 + (e & 15)];
#if ORACLE_MUTANT == 10
    const int nib = e < 16 ? (byte >> 4) : (byte & 15); /* mutant: nibble halves swapped */
#else
    const int nib = e < 16 ? (byte & 15) : (byte >> 4);
#endif
#if ORACLE_MUTANT == 9
    const int hb = (int)((qh >> (31 - e)) & 1u); /* mutant: qh bit order reversed */
#else
    const int hb = (int)((qh >> e) & 1u);
#endif
    const int q = nib | (hb << 4);
#if ORACLE_MUTANT == 11
    return q; /* mutant: the -16 offset dropped */
#else
    return q - 16;
#endif
}

/* Decoded Q5_0 weights as int8: w [rows, K] = q - 16 in [-16, 15]. */
void oracle_decode_q5_0(const uint8_t* w5, int8_t* w, int64_t rows, int64_t K) {
    const int64_t KB = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < KB; ++b) {
            const uint8_t* blk = w5 + (r * KB + b) * Q50_BYTES;
            for (int e = 0; e < QK; ++e) w[r * K + b * QK + e] = (int8_t)q50_value(blk, e);
        }
}

/* Integer block sums S[i, j, b] = sum_{e < 32} a[i, 32b + e] * (q[j, 32b + e] - 16), int64. */
void oracle_blocksums_q5_0(const int8_t* a, const uint8_t* w5, int64_t* S, int64_t M, int64_t N, int64_t K) {
    const int64_t KB = K / QK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            for (int64_t b = 0; b < KB; ++b) {
                const uint8_t* blk = w5 + (j * KB + b) * Q50_BYTES;
                int64_t acc = 0;
                for (int e = 0; e < QK; ++e) acc += (int64_t)a[i * K + b * QK + e] * (int64_t)q50_value(blk, e);
                S[(i * N + j) * KB + b] = acc;
            }
}

/* q50_qdot_t in double, with the same tolerance as qdot_t: out[i, j] =
 * sum_b as[i, b] * ws(j, b) * S[i, j, b]; bound = 1e-5 * sum_b |t_b| + 1e-6. */
void oracle_qdot_q5_0(const int8_t* a, const float* as, const uint8_t* w5, const float* ws,
                      double* out, double* bound, int64_t M, int64_t N, int64_t K, int ws_layout) {
    const int64_t KB = K / QK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double T = 0.0, U = 0.0;
            for (int64_t b = 0; b < KB; ++b) {
                const uint8_t* blk = w5 + (j * KB + b) * Q50_BYTES;
                int64_t S = 0;
                for (int e = 0; e < QK; ++e) S += (int64_t)a[i * K + b * QK + e] * (int64_t)q50_value(blk, e);
                const double wsb = ws_layout ? (double)ws[b * N + j] : (double)ws[j * KB + b];
                const double t = (double)as[i * KB + b] * wsb * (double)S;
                T += t;
                U += fabs(t);
            }
            out[i * N + j] = T;
            if (bound) bound[i * N + j] = 1e-5 * U + 1e-6;
        }
}
