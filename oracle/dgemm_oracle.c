/*
 * dgemm_oracle.c -- the oracle for the dense GEMM hot path.
 *
 * TEST INFRASTRUCTURE. This file is a plain, slow, obviously correct CPU
 * restatement of what the GPU library computes, in float64. Only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark load it; the
 * library never does, and it shares no code, header or table with the CUDA
 * sources. Every loop below is the textbook definition; there is no blocking,
 * no fusion and no reordering beyond choosing the loop order that walks memory
 * contiguously.
 *
 * Sources (web pages describing the method; cited by page title and section):
 *  [W1] DeepGEMM write-up, czchanglian.com/news/51329
 *  [W3] "DeepGEMM: FP8 Tensor Core GEMM", bjdmk.com.cn/news/6078902
 *
 * Readings where the pages are silent:
 *  - beta == 0 means C is not read (BLAS convention).
 *  - E4M3 is the "fn" variant: bias 7, no infinities, S.1111.111 is NaN, max
 *    finite 448 (the per-row scale amax/448 of the workloads pins max = 448).
 *  - Rounding to E4M3 and BF16 is round-to-nearest, ties to even; E4M3
 *    saturates to +-448 instead of overflowing.
 *  - A row whose amax is 0 gets scale 1.0 and all-zero codes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORC_F64 0
#define ORC_F32 1
#define ORC_BF16 2
#define ORC_E4M3 3

/* ---- scalar codecs ---------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32 word. */
double orc_bf16_to_f64(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits ([W3] §1.2).
 * Exponent field 0 holds the subnormals m/8 * 2^-6. */
double orc_e4m3_to_f64(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest finite E4M3 value; on a tie take the code whose
 * mantissa LSB is 0; magnitudes above 448 saturate to 448. Written as a search
 * over the 127 non-negative finite codes, whose values increase with the code. */
uint8_t orc_f64_to_e4m3(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;            /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_to_f64((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    double vlo = orc_e4m3_to_f64((uint8_t)lo), vhi = orc_e4m3_to_f64((uint8_t)hi);
    int pick;
    if (a - vlo < vhi - a) pick = lo;
    else if (a - vlo > vhi - a) pick = hi;
    else pick = (lo & 1) ? hi : lo;   /* tie: even mantissa */
    return (uint8_t)(sign | pick);
}

/* Round a double to the nearest BF16 value (8 significant bits, exponent range
 * of binary32, subnormal spacing 2^-133), ties to even; returned as a double. */
double orc_round_bf16(double x) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int e;
    (void)frexp(x, &e);               /* |x| = f * 2^e, f in [0.5, 1) */
    if (e < -125) e = -125;           /* below 2^-126 the spacing is fixed */
    double quantum = ldexp(1.0, e - 8);
    double r = nearbyint(x / quantum) * quantum;  /* default mode: ties to even */
    if (fabs(r) >= ldexp(1.0, 128)) return copysign(INFINITY, x);
    return r;
}

uint16_t orc_f64_to_bf16(double x) {
    float f = (float)orc_round_bf16(x);   /* exact: the value is a BF16 value */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    if (isnan(x)) return 0x7FC0;
    return (uint16_t)(w >> 16);
}

/* SiLU(y) = y * sigmoid(y) = y / (1 + e^-y). */
double orc_silu(double y) { return y / (1.0 + exp(-y)); }

/* GELU in its erf form: y/2 * (1 + erf(y / sqrt 2)). */
double orc_gelu(double y) { return 0.5 * y * (1.0 + erf(y / sqrt(2.0))); }

double orc_relu(double y) { return y > 0.0 ? y : 0.0; }

/* ---- array helpers ---------------------------------------------------- */

/* Exact widening of a raw buffer of n elements of the given type to double. */
int orc_decode(const void* src, int type, int64_t n, double* dst) {
    int64_t i;
    switch (type) {
    case ORC_F64: memcpy(dst, src, (size_t)n * sizeof(double)); return 0;
    case ORC_F32:
        for (i = 0; i < n; ++i) dst[i] = (double)((const float*)src)[i];
        return 0;
    case ORC_BF16:
        for (i = 0; i < n; ++i) dst[i] = orc_bf16_to_f64(((const uint16_t*)src)[i]);
        return 0;
    case ORC_E4M3:
        for (i = 0; i < n; ++i) dst[i] = orc_e4m3_to_f64(((const uint8_t*)src)[i]);
        return 0;
    }
    return -1;
}

/* Dequantise a rows x cols matrix stored row-major: X[r][c] * scale[r]
 * (axis 0) or X[r][c] * scale[c] (axis 1). [W3] §3.2: the A scale is per row
 * (per token), the B scale is per output channel. */
int orc_dequant(const void* codes, int type, int64_t rows, int64_t cols,
                const float* scale, int axis, double* dst) {
    int64_t r, c;
    if (orc_decode(codes, type, rows * cols, dst) != 0) return -1;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            dst[r * cols + c] *= (double)(axis == 0 ? scale[r] : scale[c]);
    return 0;
}

/* Per-group dequantisation: the scales change along K every `group` elements.
 * codes is a rows x cols row-major matrix of E4M3 codes; k_axis says which of
 * its two indices runs along K (1: the column index, as in A [M,K] or B stored
 * [N,K]; 0: the row index, as in B stored [K,N]). The other index i (a token or
 * an output channel) selects the scale within a group:
 *     dst[r][c] = dec(codes[r][c]) * scale[(k / group) * L + i],
 * with (k, i) = (c, r) when k_axis == 1 and (r, c) when k_axis == 0, and
 * L = the extent of i. The scale table is group-major: for group j, the L
 * scales of that K group are contiguous. This is the per-group scale
 * granularity the FP8 page asks integrators to confirm ([W3] §3.2), as
 * opposed to one scale per row or channel for the whole of K. */
int orc_dequant_grouped(const uint8_t* codes, int64_t rows, int64_t cols, const float* scale,
                        int k_axis, int64_t group, double* dst) {
    int64_t r, c;
    const int64_t L = k_axis ? rows : cols;
    if (group <= 0 || (k_axis != 0 && k_axis != 1)) return -1;
    if (orc_decode(codes, ORC_E4M3, rows * cols, dst) != 0) return -1;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c) {
            const int64_t k = k_axis ? c : r;
            const int64_t i = k_axis ? r : c;
            dst[r * cols + c] *= (double)scale[(k / group) * L + i];
        }
    return 0;
}

/* out[(i - row0) * N + n] = alpha * sum_k a(i,k) * b(k,n) + beta * c(i,n)
 * for rows i in [row0, row1). [W1] §1.1: C = alpha*A*B + beta*C, A is MxK,
 * B is KxN. b(k,n) is B[k*N + n] when b_nk == 0 (B stored KxN) and B[n*K + k]
 * when b_nk == 1 (B stored NxK, the weight layout of a linear layer).
 * C (MxN, row-major) is read only when beta != 0. */
int orc_gemm(const double* A, const double* B, int b_nk, const double* C,
             double alpha, double beta, int64_t M, int64_t N, int64_t K,
             int64_t row0, int64_t row1, double* out, int nthreads) {
    int64_t i;
    if (row0 < 0 || row1 > M || row0 > row1) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
    for (i = row0; i < row1; ++i) {
        double* o = out + (i - row0) * N;
        int64_t n, k;
        if (!b_nk) {
            for (n = 0; n < N; ++n) o[n] = 0.0;
            for (k = 0; k < K; ++k) {
                double a = A[i * K + k];
                const double* b = B + k * N;
                for (n = 0; n < N; ++n) o[n] += a * b[n];
            }
        } else {
            for (n = 0; n < N; ++n) {
                double s = 0.0;
                const double* a = A + i * K;
                const double* b = B + n * K;
                for (k = 0; k < K; ++k) s += a[k] * b[k];
                o[n] = s;
            }
        }
        for (n = 0; n < N; ++n) {
            o[n] *= alpha;
            if (beta != 0.0) o[n] += beta * C[i * N + n];
        }
    }
    return 0;
}

/* Fused epilogue on rows x N values ([W1] §6.1): y = x + bias[n], then the
 * activation (0 none, 1 ReLU, 2 GELU, 3 SiLU). bias may be NULL. */
int orc_epilogue(double* X, int64_t rows, int64_t N, const float* bias, int act) {
    int64_t r, n;
    for (r = 0; r < rows; ++r)
        for (n = 0; n < N; ++n) {
            double y = X[r * N + n] + (bias ? (double)bias[n] : 0.0);
            switch (act) {
            case 0: break;
            case 1: y = orc_relu(y); break;
            case 2: y = orc_gelu(y); break;
            case 3: y = orc_silu(y); break;
            default: return -1;
            }
            X[r * N + n] = y;
        }
    return 0;
}

/* Per-row (per-token) output quantisation ([W1] §6.2, with E4M3 codes and no
 * zero point): s[r] = max_n |z[r][n]| / 448 and q[r][n] = RN_E4M3(z / s[r]). */
int orc_requant_rows(const double* Z, int64_t rows, int64_t N, uint8_t* q, double* s) {
    int64_t r, n;
    for (r = 0; r < rows; ++r) {
        double amax = 0.0, sr;
        for (n = 0; n < N; ++n) {
            double a = fabs(Z[r * N + n]);
            if (a > amax) amax = a;
        }
        sr = amax > 0.0 ? amax / 448.0 : 1.0;
        s[r] = sr;
        for (n = 0; n < N; ++n)
            q[r * N + n] = amax > 0.0 ? orc_f64_to_e4m3(Z[r * N + n] / sr) : 0;
    }
    return 0;
}

/* Vectorised codec entry points for the tests. */
void orc_encode_e4m3_array(const double* x, int64_t n, uint8_t* q) {
    int64_t i;
    for (i = 0; i < n; ++i) q[i] = orc_f64_to_e4m3(x[i]);
}

void orc_round_bf16_array(const double* x, int64_t n, double* y) {
    int64_t i;
    for (i = 0; i < n; ++i) y[i] = orc_round_bf16(x[i]);
}

void orc_encode_bf16_array(const double* x, int64_t n, uint16_t* y) {
    int64_t i;
    for (i = 0; i < n; ++i) y[i] = orc_f64_to_bf16(x[i]);
}
