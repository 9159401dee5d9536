/*
 * oracle/mx_quant.c -- plain fp64 reference for MXFP8 block quantisation.
 *
 * TEST INFRASTRUCTURE.  This file is part of the CPU oracle.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the CUDA
 * library never does, and this file shares no code with it.
 *
 * What it follows (Fish Audio, "How we made our TTS API free", p2 section
 * "Estrategia de cuantizacion FP8", and the copy on X, section "Custom kernels
 * for the shapes TTS actually uses"): mxfp8 is 1x32 microscaling in the OCP MX
 * format -- every 32 consecutive elements along K share one power-of-two
 * scale stored as a UE8M0 byte, and each element is an OCP FP8 E4M3 number.
 * The pages give no rounding or scale rule; the OCP MX rule is used:
 *
 *   scale exponent  e = floor(log2(amax)) - 8      (8 = emax of E4M3)
 *   UE8M0 byte        = e + 127, e clamped to [-127, 127]; amax == 0 -> byte 0
 *   element code      = E4M3 round-to-nearest-even of v * 2^-e, saturating
 *                       magnitudes above 448 to 448; the sign is kept, so a
 *                       negative value that rounds to zero is 0x80.
 *
 * Everything here is done in double precision with plain loops.  floor(log2)
 * is taken from frexp (exact for every finite input, subnormals included),
 * never from log2().  Scaling by 2^-e is exact in double.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- E4M3
 * OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN.  Code c (7 magnitude
 * bits, 0..126) has exponent field E = c >> 3 and mantissa m = c & 7:
 *   E == 0 : subnormal, value m/8 * 2^(1-7) = m * 2^-9
 *   E >= 1 : normal,    value (1 + m/8) * 2^(E-7)
 * Values grow with the code, so the table is sorted.
 */
double mxo_e4m3_value(int c)
{
    int E = c >> 3, m = c & 7;
    if (E == 0) return ldexp((double)m, -9);
    return ldexp(1.0 + m / 8.0, E - 7);
}

/* Nearest E4M3 magnitude code to t >= 0; ties go to the even code (mantissa
 * LSB 0); t above the largest finite value 448 (code 126) saturates. */
int mxo_e4m3_round(double t)
{
    if (t >= 448.0) return 126;
    /* largest code lo with value(lo) <= t (binary search over 0..126) */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (mxo_e4m3_value(mid) <= t) lo = mid; else hi = mid;
    }
    if (mxo_e4m3_value(hi) <= t) lo = hi;
    if (lo == 126) return 126;
    double below = mxo_e4m3_value(lo), above = mxo_e4m3_value(lo + 1);
    double d_below = t - below, d_above = above - t;   /* both exact */
    if (d_below < d_above) return lo;
    if (d_above < d_below) return lo + 1;
    return (lo & 1) ? lo + 1 : lo;                      /* tie: even code */
}

/* ---------------------------------------------------------------- UE8M0 */
/* The block exponent e for a block whose largest magnitude is amax. */
int mxo_block_exponent(double amax)
{
    if (amax == 0.0) return -127;
    int ex;
    frexp(amax, &ex);          /* amax = f * 2^ex, f in [0.5, 1) */
    int e = (ex - 1) - 8;      /* floor(log2(amax)) - emax(E4M3) */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Quantise one block of n (= 32) values. */
static void quantize_block(const double *v, int n, uint8_t *codes, uint8_t *scale)
{
    double amax = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(v[i]);
        if (a > amax) amax = a;
    }
    int e = mxo_block_exponent(amax);
    *scale = (uint8_t)(e + 127);
    for (int i = 0; i < n; ++i) {
        double t = ldexp(fabs(v[i]), -e);
        int c = mxo_e4m3_round(t);
        codes[i] = (uint8_t)(c | (signbit(v[i]) ? 0x80 : 0));
    }
}

/* v [rows, K] (row stride K) -> codes [rows, K], scales [rows, K/32]
 * (row-major: the K-block index runs fastest).  K must be a multiple of 32. */
void mxo_quantize_f64(const double *v, long rows, long K, uint8_t *codes, uint8_t *scales)
{
    long nb = K / 32;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r)
        for (long b = 0; b < nb; ++b)
            quantize_block(v + r * K + b * 32, 32, codes + r * K + b * 32, scales + r * nb + b);
}

/* Same, for bf16 inputs given as their 16-bit patterns (each is widened to
 * the exactly equal double first). */
void mxo_quantize_bf16(const uint16_t *bits, long rows, long K, uint8_t *codes, uint8_t *scales)
{
    long nb = K / 32;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double blk[32];
        for (long b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i) {
                uint32_t w = (uint32_t)bits[r * K + b * 32 + i] << 16;
                float f;
                memcpy(&f, &w, 4);
                blk[i] = (double)f;
            }
            quantize_block(blk, 32, codes + r * K + b * 32, scales + r * nb + b);
        }
    }
}

/* codes [rows, K] + row-major scales [rows, K/32] -> exact values [rows, K]. */
void mxo_dequantize(const uint8_t *codes, const uint8_t *scales, long rows, long K, double *out)
{
    long nb = K / 32;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r)
        for (long k = 0; k < K; ++k) {
            uint8_t c = codes[r * K + k];
            double mag = mxo_e4m3_value(c & 0x7F);
            int e = (int)scales[r * nb + k / 32] - 127;
            double val = ldexp(mag, e);
            out[r * K + k] = (c & 0x80) ? -val : val;
        }
}

/* ---------------------------------------------------------------- bf16
 * Round each double to the nearest bf16 value (8 significant bits, exponent
 * range of float32), ties to even, in one step (no detour through float32,
 * which could round twice).  Returns the 16-bit patterns.  Inputs are finite
 * and below the bf16 overflow threshold. */
void mxo_round_bf16(const double *y, long n, uint16_t *out)
{
    for (long i = 0; i < n; ++i) {
        double a = fabs(y[i]);
        double r;
        if (a == 0.0) {
            r = 0.0;
        } else {
            int ex;
            frexp(a, &ex);                  /* a in [2^(ex-1), 2^ex) */
            int q = ex - 8;                 /* quantum 2^(ex-1-7) */
            if (q < -133) q = -133;         /* bf16 subnormal quantum */
            r = ldexp(nearbyint(ldexp(a, -q)), q);   /* round-half-even */
        }
        float f = (float)r;                  /* exact: r is a bf16 value */
        uint32_t w;
        memcpy(&w, &f, 4);
        out[i] = (uint16_t)((w >> 16) | (signbit(y[i]) ? 0x8000u : 0u));
    }
}
