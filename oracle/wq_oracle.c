/*
 * wq_oracle.c -- plain, slow, fp64 CPU oracle for weight-only quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library under
 * weight_only_quantized_wq_gb300/ may include, link or call this file.  Only
 * tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
 * load it (through oracle/__init__.py).  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * What it computes (each function cites the passage it follows):
 *
 *   BitDistiller, quantization/triton_kernels.py, quant_matmul_kernel
 *   (docstring and the K loop):
 *     a (M,K); qw (K/pack_num, N) int32; scales (K/group_size, N);
 *     qzeros (K/group_size/pack_num, N) int32; pack_num = 32 / w_bit.
 *     code(k,n) = (qw[k/pack_num][n] >> ((k % pack_num) * w_bit)) & offset,
 *     offset = 2^w_bit - 1.
 *   The page is cut off before the scale/zero step.  Reading taken here:
 *     w(k,n) = (code(k,n) - zero(g,n)) * scale(g,n), g = k / group_size,
 *     zero(g,n) unpacked from qzeros exactly like the weights but along the
 *     group axis, with ceil(G / pack_num) rows; a NULL qzeros means the
 *     symmetric case with zero = 2^(w_bit-1) (8 for int4, as in Marlin's
 *     dequant(), aphrodite-engine marlin_cuda_kernel.cu, which folds "-8").
 *   y(m,n) = sum_k x(m,k) * w(k,n), in fp64, k ascending.
 *
 *   tiny-llm, kernels/int8_gemv.py, int8_matmul docstring:
 *     x (M,K) bf16/fp16; q (N,K) int8; scale (N,) fp32 -> y (M,N) fp32,
 *     y(m,n) = scale(n) * sum_k x(m,k) * q(n,k).
 *
 * Half and bfloat16 inputs are decoded bit by bit (IEEE binary16 and the
 * truncated-binary32 bfloat16 format); no compiler half type is used.
 *
 * Return value of every entry point: 0 on success, -1 on an invalid argument.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double wq_oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero / subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of binary32 -- 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double wq_oracle_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* f * 2^-7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* binary32 from its bit pattern, done by hand like the two above. */
double wq_oracle_f32_to_f64(uint32_t b)
{
    int sign = (b >> 31) & 1;
    int e = (b >> 23) & 0xff;
    uint32_t f = b & 0x7fffffu;
    double v;
    if (e == 0)
        v = ldexp((double)f, -149);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x800000u + f), e - 150);
    return sign ? -v : v;
}

static double decode16(uint16_t h, int is_bf16)
{
    return is_bf16 ? wq_oracle_bf16_to_f64(h) : wq_oracle_f16_to_f64(h);
}

/* Array form of the two decoders above, for the exhaustive decoder pins. */
int wq_oracle_decode16_array(const uint16_t *in, size_t n, int is_bf16, double *out)
{
    if (!in || !out) return -1;
    for (size_t i = 0; i < n; ++i) out[i] = decode16(in[i], is_bf16);
    return 0;
}

static int valid_wbit(int w_bit) { return w_bit == 2 || w_bit == 4 || w_bit == 8; }

/* One w_bit-wide field of a packed word: logical shift of the unsigned word,
 * then the mask (the page shifts a signed int32, which only matters above
 * the mask; an unsigned shift gives the same field). */
static uint32_t field(uint32_t word, int slot, int w_bit)
{
    uint32_t mask = (1u << w_bit) - 1u;
    return (word >> (slot * w_bit)) & mask;
}

/* Page-2 weight layout -> codes (K, N) row-major, one byte per code.
 * BitDistiller quant_matmul_kernel: qw_offs = (k // pack_num) * N + n,
 * then (packed >> ((k % pack_num) * w_bit)) & offset. */
int wq_oracle_unpack(const uint32_t *qw, int K, int N, int w_bit, uint8_t *codes)
{
    if (!qw || !codes || K < 0 || N < 0 || !valid_wbit(w_bit)) return -1;
    int pack = 32 / w_bit;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n)
            codes[(size_t)k * N + n] =
                (uint8_t)field(qw[(size_t)(k / pack) * N + n], k % pack, w_bit);
    return 0;
}

/* Inverse of wq_oracle_unpack: codes (K, N) -> qw (ceil(K/pack), N).
 * Fields past K in the last row are left 0.  Codes wider than w_bit are an error. */
int wq_oracle_pack(const uint8_t *codes, int K, int N, int w_bit, uint32_t *qw)
{
    if (!qw || !codes || K < 0 || N < 0 || !valid_wbit(w_bit)) return -1;
    int pack = 32 / w_bit;
    int rows = (K + pack - 1) / pack;
    for (size_t i = 0; i < (size_t)rows * N; ++i) qw[i] = 0;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            uint32_t c = codes[(size_t)k * N + n];
            if (c >> w_bit) return -1;
            qw[(size_t)(k / pack) * N + n] |= c << ((k % pack) * w_bit);
        }
    return 0;
}

/* Zero point of group g, column n.  qzeros is packed along the group axis,
 * LSB first, exactly like the weights along K (reading of the page's
 * "qzeros: (K // group_size // pack_num, N)"; rows = ceil(G / pack_num)). */
static double zero_of(const uint32_t *qzeros, int g, int n, int N, int w_bit)
{
    if (!qzeros) return (double)(1 << (w_bit - 1));
    int pack = 32 / w_bit;
    return (double)field(qzeros[(size_t)(g / pack) * N + n], g % pack, w_bit);
}

/* Dequantized weight matrix w (K, N) in fp64: (code - zero) * scale.
 * group_size <= 0 or == K means one group per column (per-channel). */
int wq_oracle_dequant(const uint32_t *qw, const uint16_t *scales, int s_is_bf16,
                      const uint32_t *qzeros, int K, int N, int w_bit,
                      int group_size, double *w)
{
    if (!qw || !scales || !w || K <= 0 || N < 0 || (w_bit != 2 && w_bit != 4)) return -1;
    if (group_size <= 0) group_size = K;
    if (K % group_size) return -1;
    int pack = 32 / w_bit;
    for (int k = 0; k < K; ++k) {
        int g = k / group_size;
        for (int n = 0; n < N; ++n) {
            double q = (double)field(qw[(size_t)(k / pack) * N + n], k % pack, w_bit);
            double z = zero_of(qzeros, g, n, N, w_bit);
            double s = decode16(scales[(size_t)g * N + n], s_is_bf16);
            w[(size_t)k * N + n] = (q - z) * s;
        }
    }
    return 0;
}

/* Grouped weight-only matmul, fp64.
 *   x       (M, K) fp16 (x_is_bf16 = 0) or bf16 (1), row-major
 *   qw      (K/pack, N) int32, page-2 layout
 *   scales  (K/group_size, N) fp16 or bf16
 *   qzeros  (ceil(G/pack), N) int32 or NULL (symmetric, zero = 2^(w_bit-1))
 * Computes only rows rows[0..nrows) (all rows if rows == NULL, nrows = M)
 * and columns [n0, n1).  y is (nrows, n1 - n0) row-major fp64.
 * For each output the sum runs over k in ascending order. */
int wq_oracle_matmul_grouped(const uint16_t *x, int x_is_bf16, const uint32_t *qw,
                             const uint16_t *scales, int s_is_bf16,
                             const uint32_t *qzeros, int M, int N, int K,
                             int w_bit, int group_size, int n0, int n1,
                             const int32_t *rows, int nrows, double *y)
{
    if (!x || !qw || !scales || !y || M < 0 || N < 0 || K <= 0) return -1;
    if (w_bit != 2 && w_bit != 4) return -1;
    if (group_size <= 0) group_size = K;
    if (K % group_size) return -1;
    if (n0 < 0 || n1 > N || n0 > n1) return -1;
    if (!rows) nrows = M;
    if (nrows < 0) return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= M)) return -1;

    int pack = 32 / w_bit;
    int width = n1 - n0;
    double *wrow = (double *)malloc(sizeof(double) * (width > 0 ? width : 1));
    if (!wrow) return -1;
    for (size_t i = 0; i < (size_t)nrows * width; ++i) y[i] = 0.0;

    for (int k = 0; k < K; ++k) {
        int g = k / group_size;
        /* row k of the dequantized weight, columns [n0, n1) */
        for (int j = 0; j < width; ++j) {
            int n = n0 + j;
            double q = (double)field(qw[(size_t)(k / pack) * N + n], k % pack, w_bit);
            double z = zero_of(qzeros, g, n, N, w_bit);
            double s = decode16(scales[(size_t)g * N + n], s_is_bf16);
            wrow[j] = (q - z) * s;
        }
        for (int r = 0; r < nrows; ++r) {
            int m = rows ? rows[r] : r;
            double xv = decode16(x[(size_t)m * K + k], x_is_bf16);
            double *yr = y + (size_t)r * width;
            for (int j = 0; j < width; ++j) yr[j] += xv * wrow[j];
        }
    }
    free(wrow);
    return 0;
}

/* int8 weight-only per-output-channel matmul, fp64 (tiny-llm int8_matmul):
 *   x (M, K) fp16/bf16; q (N, K) int8, K contiguous; scale (N,) fp32 bits.
 *   y(m, n) = scale(n) * sum_k x(m, k) * q(n, k).
 * Same row / column selection and output layout as the grouped oracle. */
int wq_oracle_matmul_int8(const uint16_t *x, int x_is_bf16, const int8_t *q,
                          const uint32_t *scale_bits, int M, int N, int K,
                          int n0, int n1, const int32_t *rows, int nrows, double *y)
{
    if (!x || !q || !scale_bits || !y || M < 0 || N < 0 || K <= 0) return -1;
    if (n0 < 0 || n1 > N || n0 > n1) return -1;
    if (!rows) nrows = M;
    if (nrows < 0) return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= M)) return -1;
    int width = n1 - n0;
    for (int r = 0; r < nrows; ++r) {
        int m = rows ? rows[r] : r;
        for (int j = 0; j < width; ++j) {
            int n = n0 + j;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += decode16(x[(size_t)m * K + k], x_is_bf16) * (double)q[(size_t)n * K + k];
            y[(size_t)r * width + j] = wq_oracle_f32_to_f64(scale_bits[n]) * acc;
        }
    }
    return 0;
}

/*
 * Liger kernels, ops/experimental/mm_int8int2.py (page 1): ternary weights in
 * {-1, 0, 1} stored plus one as 2-bit fields of uint8, planar along K.
 * pack_weights / unpack_weights: with R = K / 4 rows of bytes (K % 4 == 0
 * here), plane i = 0..3 holds rows k = i R .. i R + R - 1 in bits 2i, 2i+1
 * of byte [k - i R][n], i.e. for any k:
 *   w(k, n) = ((packed[k mod R][n] >> (2 (k div R))) & 3) - 1.
 * matmul_kernel: C = A (M, K) int8 times w (K, N), accumulated in int32.
 * Here the sum is exact in int64 (the caller checks it fits int32).
 */
static int t2_value(const uint8_t *packed, int K, int N, int k, int n)
{
    int R = K / 4;
    return (int)((packed[(size_t)(k % R) * N + n] >> (2 * (k / R))) & 3u) - 1;
}

/* Planar packed bytes (K/4, N) -> weights (K, N) as int8 in {-1, 0, 1, 2}. */
int wq_oracle_t2_unpack(const uint8_t *packed, int K, int N, int8_t *w)
{
    if (!packed || !w || K <= 0 || N < 0 || K % 4) return -1;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n)
            w[(size_t)k * N + n] = (int8_t)t2_value(packed, K, N, k, n);
    return 0;
}

/* Inverse: weights (K, N) in {-1, 0, 1, 2} -> planar packed bytes (K/4, N). */
int wq_oracle_t2_pack(const int8_t *w, int K, int N, uint8_t *packed)
{
    if (!packed || !w || K <= 0 || N < 0 || K % 4) return -1;
    int R = K / 4;
    for (size_t i = 0; i < (size_t)R * N; ++i) packed[i] = 0;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            int v = w[(size_t)k * N + n] + 1;
            if (v < 0 || v > 3) return -1;
            packed[(size_t)(k % R) * N + n] |= (uint8_t)(v << (2 * (k / R)));
        }
    return 0;
}

/* y (M, N) int64 = x (M, K) int8 times the unpacked weights, k ascending. */
int wq_oracle_t2_matmul(const int8_t *x, const uint8_t *packed, int M, int N, int K, int64_t *y)
{
    if (!x || !packed || !y || M < 0 || N < 0 || K <= 0 || K % 4) return -1;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k)
                acc += (int64_t)x[(size_t)m * K + k] * (int64_t)t2_value(packed, K, N, k, n);
            y[(size_t)m * N + n] = acc;
        }
    return 0;
}
