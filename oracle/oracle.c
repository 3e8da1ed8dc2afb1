/*
 * oracle.c -- plain, slow CPU oracle for the asymmetric group-wise W4A16 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file:
 * it is used by tests/, by __graft_entry__.smoke() and by the cpu_baseline leg of bench.py.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (all floating point in IEEE double):
 *   y[m][n] = sum_k x[m][k] * W[k][n],      W[k][n] = (q[k][n] - z[k/g][n]) * s[k/g][n]
 * with 4-bit codes q, z in 0..15 and fp16 scales s.
 *
 * Sources, by page:
 *  - "Carga de capas cuantizadas: AWQ / GPTQ / Marlin / fp8" (vLLM architecture walkthrough),
 *    section "Flujo de datos": qweight int32 [K, N/8] and qzeros int32 [K/g, N/8] packed along
 *    the output dimension (packed_dim=1, pack_factor 8), scales [K/g, N], num_groups = K // g.
 *    Section "Motivacion de diseno": AWQ packs in a non-standard order along the output
 *    dimension; the GPTQ-style "standard" format packs along the input dimension in plain bit
 *    order.  Section "Limites y fallos": group_size = -1 means one group over all of K.
 *  - vllm-omni commit "Add cpu_int4, an asymmetric 4-bit weight path for vLLM's CPU backend":
 *    the grid is asymmetric (a zero point per group and channel, sym=False), group-wise.
 *  - vllm-omni commit "cpu_int4: dequantize prefill weights from the tinygemm layout, not a
 *    copy": the CPU kernel's [N/64][K][32 bytes] layout, byte d of each 32-byte run holding
 *    channel d in its low nibble and channel d+32 in its high nibble.
 *  - vllm-omni commit "cpu_int4: repack weights in n-blocks, to bound the load-time peak":
 *    n-blocks of that layout are independent, so packing can run one n-chunk at a time and
 *    must give the same bytes as packing the whole matrix.
 *
 * Readings taken where the pages are silent:
 *  - the dequant formula W = (q - z) * s with the raw stored zero z (no +1 offset);
 *  - the AWQ slot order: nibble slot j (bits 4j..4j+3, counted from the least significant bit
 *    of the word read as unsigned 32-bit) holds column 8c + {0,2,4,6,1,3,5,7}[j];
 *  - group of row k is floor(k / g), groups contiguous along K;
 *  - the fp16 result of a dequantized weight is the single round-to-nearest-even rounding of
 *    the exact product (no flush to zero).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* AWQ nibble slot j -> column offset inside the 8-column word. */
static const int awq_slot_to_col[8] = {0, 2, 4, 6, 1, 3, 5, 7};

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- IEEE binary16 --------- */

/* Exact value of an IEEE binary16 bit pattern. */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even, with gradual underflow and
 * overflow to infinity.  Written from the definition of the format. */
uint16_t oracle_double_to_half(double v) {
    if (isnan(v)) return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7c00;
    int e2;
    frexp(a, &e2);              /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;             /* a in [2^E, 2^(E+1)) */
    if (E > 15) return sign | 0x7c00;
    int qexp = (E >= -14) ? (E - 10) : -24;       /* spacing of binary16 values near a */
    double scaled = ldexp(a, -qexp);                /* exact: power-of-two scaling */
    double S = floor(scaled);
    double rem = scaled - S;                        /* exact: scaled < 2^12 */
    if (rem > 0.5 || (rem == 0.5 && fmod(S, 2.0) != 0.0)) S += 1.0;
    if (E < -14) {
        /* subnormal range: S in [0, 1024]; S == 1024 is the smallest normal, whose bit
         * pattern 0x0400 equals S, so the encoding carries over by itself. */
        return sign | (uint16_t)S;
    }
    if (S >= 2048.0) {          /* rounding carried into the next binade */
        S = 1024.0;
        E += 1;
        if (E > 15) return sign | 0x7c00;
    }
    return sign | (uint16_t)(((E + 15) << 10) | ((int)S - 1024));
}

void oracle_double_to_half_array(const double *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_half(in[i]);
}

void oracle_half_to_double_array(const uint16_t *in, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(in[i]);
}

/* ---------------------------------------------------------------- bfloat16 -------------- */
/* The bf16 variant of the layer (activations, scales and output in bfloat16: the CPU path of
 * vllm-omni commit "Add cpu_int4 ..." runs in bf16).  bfloat16: 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits, gradual underflow. */

/* Exact value of a bfloat16 bit pattern. */
double oracle_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-133 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to even, with gradual underflow and overflow to
 * infinity (same construction as the binary16 rounding above, with bfloat16's parameters). */
uint16_t oracle_double_to_bf16(double v) {
    if (isnan(v)) return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7f80;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;                                 /* a in [2^E, 2^(E+1)) */
    if (E > 127) return sign | 0x7f80;
    int qexp = (E >= -126) ? (E - 7) : -133;        /* spacing of bfloat16 values near a */
    double scaled = ldexp(a, -qexp);
    double S = floor(scaled);
    double rem = scaled - S;
    if (rem > 0.5 || (rem == 0.5 && fmod(S, 2.0) != 0.0)) S += 1.0;
    if (E < -126) return sign | (uint16_t)S;        /* S == 128 is the smallest normal, 0x0080 */
    if (S >= 256.0) {
        S = 128.0;
        E += 1;
        if (E > 127) return sign | 0x7f80;
    }
    return sign | (uint16_t)(((E + 127) << 7) | ((int)S - 128));
}

void oracle_double_to_bf16_array(const double *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(in[i]);
}

/* ---------------------------------------------------------------- AWQ packing ----------- */

/* Unpack AWQ-packed codes: packed int32 [rows][N/8] -> codes uint8 [rows][N].
 * Used for qweight (rows = K) and for qzeros (rows = K/g). */
void oracle_awq_unpack(const int32_t *packed, int rows, int N, uint8_t *codes) {
    int C = N / 8;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < C; ++c) {
            uint32_t w = (uint32_t)packed[(int64_t)r * C + c];
            for (int j = 0; j < 8; ++j)
                codes[(int64_t)r * N + 8 * c + awq_slot_to_col[j]] = (uint8_t)((w >> (4 * j)) & 0xFu);
        }
}

/* Inverse of oracle_awq_unpack. */
void oracle_awq_pack(const uint8_t *codes, int rows, int N, int32_t *packed) {
    int C = N / 8;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < C; ++c) {
            uint32_t w = 0;
            for (int j = 0; j < 8; ++j)
                w |= ((uint32_t)codes[(int64_t)r * N + 8 * c + awq_slot_to_col[j]] & 0xFu) << (4 * j);
            packed[(int64_t)r * C + c] = (int32_t)w;
        }
}

/* ---------------------------------------------------------------- dequantization -------- */

typedef double (*decode16_fn)(uint16_t);

/* W[k][n] = (q[k][n] - z[k/g][n]) * s[k/g][n], exact in double, s decoded by `dec`. */
static void dequant_codes_dec(const uint8_t *q, const uint8_t *z, const uint16_t *s,
                              int K, int N, int g, decode16_fn dec, double *W) {
    for (int k = 0; k < K; ++k) {
        int G = k / g;
        for (int n = 0; n < N; ++n) {
            double qv = (double)q[(int64_t)k * N + n];
            double zv = (double)z[(int64_t)G * N + n];
            double sv = dec(s[(int64_t)G * N + n]);
            W[(int64_t)k * N + n] = (qv - zv) * sv;
        }
    }
}

/* W[k][n] = (q[k][n] - z[k/g][n]) * s[k/g][n], exact in double (fp16 scales). */
void oracle_dequant_codes_f64(const uint8_t *q, const uint8_t *z, const uint16_t *s,
                              int K, int N, int g, double *W) {
    dequant_codes_dec(q, z, s, K, N, g, oracle_half_to_double, W);
}

/* Dequantize straight from the AWQ tensors (qweight [K][N/8], qzeros [K/g][N/8],
 * scales fp16 [K/g][N]) to double W[K][N].  Returns 0, or -1 if memory ran out. */
int oracle_dequant_awq_f64(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                           int K, int N, int g, double *W) {
    int groups = K / g;
    uint8_t *q = (uint8_t *)malloc((size_t)K * N);
    uint8_t *z = (uint8_t *)malloc((size_t)groups * N);
    if (!q || !z) { free(q); free(z); return -1; }
    oracle_awq_unpack(qweight, K, N, q);
    oracle_awq_unpack(qzeros, groups, N, z);
    oracle_dequant_codes_f64(q, z, scales, K, N, g, W);
    free(q);
    free(z);
    return 0;
}

/* The fp16 weight: one round-to-nearest-even of the exact product. */
int oracle_dequant_awq_f16(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                           int K, int N, int g, uint16_t *W16) {
    int64_t n = (int64_t)K * N;
    double *W = (double *)malloc((size_t)n * sizeof(double));
    if (!W) return -1;
    if (oracle_dequant_awq_f64(qweight, qzeros, scales, K, N, g, W)) { free(W); return -1; }
    oracle_double_to_half_array(W, n, W16);
    free(W);
    return 0;
}

/* ---------------------------------------------------------------- tied embedding -------- */

/* Gather of the quantized tied embedding: the LM head's weight W [K][N] doubles as the
 * embedding table (vllm-omni commit "cpu_int4: repack weights in n-blocks, to bound the
 * load-time peak": "embedding 131072 x 2048 ... tied, so it is also the head"; commit "Add
 * cpu_int4 ...": "the quantized tied embedding").  Token t reads column n = ids[t]:
 *     out[t][k] = fp16((q[k][n] - z[k/g][n]) * s[k/g][n])     for k = 0 .. K-1,
 * the same single rounding as the dequantized weight.  Read straight from the AWQ words: the
 * code of column n sits in the nibble slot j with slot_to_col[j] == n % 8 of word n / 8.
 * An id outside [0, N) gives a row of +0.  Returns the number of such ids. */
int oracle_embed_gather(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                        int K, int N, int g, const int32_t *ids, int T, uint16_t *out) {
    int bad = 0;
    int slot_of_col[8];
    for (int j = 0; j < 8; ++j) slot_of_col[awq_slot_to_col[j]] = j;
    for (int t = 0; t < T; ++t) {
        int n = ids[t];
        uint16_t *row = out + (int64_t)t * K;
        if (n < 0 || n >= N) {
            for (int k = 0; k < K; ++k) row[k] = 0;
            ++bad;
            continue;
        }
        int word = n / 8, shift = 4 * slot_of_col[n % 8];
        for (int k = 0; k < K; ++k) {
            int G = k / g;
            uint32_t qw = (uint32_t)qweight[(int64_t)k * (N / 8) + word];
            uint32_t zw = (uint32_t)qzeros[(int64_t)G * (N / 8) + word];
            double q = (double)((qw >> shift) & 0xFu);
            double z = (double)((zw >> shift) & 0xFu);
            double sv = oracle_half_to_double(scales[(int64_t)G * N + n]);
            row[k] = oracle_double_to_half((q - z) * sv);
        }
    }
    return bad;
}

/* ---------------------------------------------------------------- the linear layer ------ */

/* y[m][n] = sum_{k=0}^{K-1} x[m][k] * W[k][n] in double, k summed in increasing order for
 * every output.  x is fp16 [M][K] row-major, W double [K][N], y double [M][N]. */
void oracle_gemm_f64(const uint16_t *x, int M, int K, const double *W, int N, double *y) {
    const int NB = 256;
    int nblocks = (N + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < nblocks; ++b) {
        int n0 = b * NB, n1 = n0 + NB < N ? n0 + NB : N;
        for (int m = 0; m < M; ++m) {
            double *yr = y + (int64_t)m * N;
            for (int n = n0; n < n1; ++n) yr[n] = 0.0;
            for (int k = 0; k < K; ++k) {
                double xv = oracle_half_to_double(x[(int64_t)m * K + k]);
                const double *Wr = W + (int64_t)k * N;
                for (int n = n0; n < n1; ++n) yr[n] += xv * Wr[n];
            }
        }
    }
}

/* The whole layer from AWQ tensors: y64 = x * W (double); y16 = fp16 rounding of y64
 * (either output may be NULL).  Returns 0, or -1 if memory ran out. */
int oracle_linear(const uint16_t *x, int M, int K, const int32_t *qweight, const int32_t *qzeros,
                  const uint16_t *scales, int N, int g, double *y64, uint16_t *y16) {
    double *W = (double *)malloc((size_t)K * N * sizeof(double));
    double *y = y64 ? y64 : (double *)malloc((size_t)M * N * sizeof(double) + 1);
    if (!W || !y) { free(W); if (!y64) free(y); return -1; }
    if (oracle_dequant_awq_f64(qweight, qzeros, scales, K, N, g, W)) {
        free(W); if (!y64) free(y); return -1;
    }
    oracle_gemm_f64(x, M, K, W, N, y);
    if (y16) oracle_double_to_half_array(y, (int64_t)M * N, y16);
    free(W);
    if (!y64) free(y);
    return 0;
}

/* Selected outputs y[m_i][n_i], each computed on its own straight from the packed AWQ words:
 * for every k the code and the zero are read out of their words scalar by scalar.
 * Used where the whole product is too large for the oracle to finish in seconds. */
void oracle_linear_sampled(const uint16_t *x, int M, int K, const int32_t *qweight,
                           const int32_t *qzeros, const uint16_t *scales, int N, int g,
                           const int64_t *m_idx, const int64_t *n_idx, int64_t count, double *out) {
    int C = N / 8;
    (void)M;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = m_idx[i], n = n_idx[i];
        int c = (int)(n / 8), j = 0;
        while (awq_slot_to_col[j] != (int)(n % 8)) ++j;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
            int G = k / g;
            uint32_t wq = (uint32_t)qweight[(int64_t)k * C + c];
            uint32_t wz = (uint32_t)qzeros[(int64_t)G * C + c];
            double qv = (double)((wq >> (4 * j)) & 0xFu);
            double zv = (double)((wz >> (4 * j)) & 0xFu);
            double sv = oracle_half_to_double(scales[(int64_t)G * N + n]);
            acc += oracle_half_to_double(x[m * K + k]) * ((qv - zv) * sv);
        }
        out[i] = acc;
    }
}

/* ---------------------------------------------------------------- other layouts --------- */

/* AWQ -> GPTQ-style standard format: qweight int32 [K/8][N] packed along the input dimension,
 * slot j = row 8r + j; qzeros int32 [K/g][N/8] packed along the output dimension in plain
 * order, slot j = column 8c + j.  Requires K % 8 == 0. */
void oracle_awq_to_standard(const int32_t *qweight_awq, const int32_t *qzeros_awq,
                            int K, int N, int g, int32_t *qweight_std, int32_t *qzeros_std) {
    int groups = K / g;
    uint8_t *q = (uint8_t *)malloc((size_t)K * N);
    uint8_t *z = (uint8_t *)malloc((size_t)groups * N);
    if (!q || !z) { free(q); free(z); return; }
    oracle_awq_unpack(qweight_awq, K, N, q);
    oracle_awq_unpack(qzeros_awq, groups, N, z);
    for (int r = 0; r < K / 8; ++r)
        for (int n = 0; n < N; ++n) {
            uint32_t w = 0;
            for (int j = 0; j < 8; ++j) w |= (uint32_t)q[(int64_t)(8 * r + j) * N + n] << (4 * j);
            qweight_std[(int64_t)r * N + n] = (int32_t)w;
        }
    for (int G = 0; G < groups; ++G)
        for (int c = 0; c < N / 8; ++c) {
            uint32_t w = 0;
            for (int j = 0; j < 8; ++j) w |= (uint32_t)z[(int64_t)G * N + 8 * c + j] << (4 * j);
            qzeros_std[(int64_t)G * (N / 8) + c] = (int32_t)w;
        }
    free(q);
    free(z);
}

/* Dequantize from the standard format, reading each code out of its word directly. */
void oracle_dequant_standard_f64(const int32_t *qweight_std, const int32_t *qzeros_std,
                                 const uint16_t *scales, int K, int N, int g, double *W) {
    for (int k = 0; k < K; ++k) {
        int G = k / g;
        for (int n = 0; n < N; ++n) {
            uint32_t wq = (uint32_t)qweight_std[(int64_t)(k / 8) * N + n];
            uint32_t wz = (uint32_t)qzeros_std[(int64_t)G * (N / 8) + n / 8];
            double qv = (double)((wq >> (4 * (k % 8))) & 0xFu);
            double zv = (double)((wz >> (4 * (n % 8))) & 0xFu);
            W[(int64_t)k * N + n] = (qv - zv) * oracle_half_to_double(scales[(int64_t)G * N + n]);
        }
    }
}

/* The CPU kernel's layout [ceil(N/64)][K][32 bytes]: in n-block b, row k, byte d holds the
 * code of channel 64b + d in its low nibble and of channel 64b + d + 32 in its high nibble.
 * Channels past N (a tail block) read as code 0.  Only n-blocks with 64b in [n0, n1) are
 * written, so a caller may pack one n-chunk at a time. */
void oracle_int4pack_cpu_chunk(const uint8_t *q, int K, int N, int n0, int n1, uint8_t *out) {
    int nblocks = (N + 63) / 64;
    for (int b = 0; b < nblocks; ++b) {
        if (64 * b < n0 || 64 * b >= n1) continue;
        for (int k = 0; k < K; ++k)
            for (int d = 0; d < 32; ++d) {
                int lo_n = 64 * b + d, hi_n = 64 * b + d + 32;
                uint8_t lo = lo_n < N ? q[(int64_t)k * N + lo_n] & 0xF : 0;
                uint8_t hi = hi_n < N ? q[(int64_t)k * N + hi_n] & 0xF : 0;
                out[((int64_t)b * K + k) * 32 + d] = (uint8_t)(lo | (hi << 4));
            }
    }
}

void oracle_int4pack_cpu(const uint8_t *q, int K, int N, uint8_t *out) {
    oracle_int4pack_cpu_chunk(q, K, N, 0, N, out);
}

/* Read the codes back out of the [N/64][K][32 bytes] layout (the de-interleave). */
void oracle_int4unpack_cpu(const uint8_t *packed, int K, int N, uint8_t *q) {
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            int b = n / 64, d = n % 64;
            uint8_t byte = packed[((int64_t)b * K + k) * 32 + (d % 32)];
            q[(int64_t)k * N + n] = d < 32 ? (byte & 0xF) : (byte >> 4);
        }
}


/* ---------------------------------------------------------------- the bf16 layer -------- */

/* As oracle_dequant_awq_f64 with bfloat16 scales. */
int oracle_dequant_awq_bf16_f64(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                                int K, int N, int g, double *W) {
    int groups = K / g;
    uint8_t *q = (uint8_t *)malloc((size_t)K * N);
    uint8_t *z = (uint8_t *)malloc((size_t)groups * N);
    if (!q || !z) { free(q); free(z); return -1; }
    oracle_awq_unpack(qweight, K, N, q);
    oracle_awq_unpack(qzeros, groups, N, z);
    dequant_codes_dec(q, z, scales, K, N, g, oracle_bf16_to_double, W);
    free(q);
    free(z);
    return 0;
}

/* The bfloat16 weight: one round-to-nearest-even of the exact product. */
int oracle_dequant_awq_bf16(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                            int K, int N, int g, uint16_t *Wb) {
    int64_t n = (int64_t)K * N;
    double *W = (double *)malloc((size_t)n * sizeof(double));
    if (!W) return -1;
    if (oracle_dequant_awq_bf16_f64(qweight, qzeros, scales, K, N, g, W)) { free(W); return -1; }
    oracle_double_to_bf16_array(W, n, Wb);
    free(W);
    return 0;
}

/* The bf16 layer: x bfloat16 [M][K], scales bfloat16; y64 = x * W in double (k summed in
 * increasing order), yb = its bfloat16 rounding (either output may be NULL).  Returns 0, or -1
 * if memory ran out. */
int oracle_linear_bf16(const uint16_t *x, int M, int K, const int32_t *qweight, const int32_t *qzeros,
                       const uint16_t *scales, int N, int g, double *y64, uint16_t *yb) {
    double *W = (double *)malloc((size_t)K * N * sizeof(double));
    double *y = y64 ? y64 : (double *)malloc((size_t)M * N * sizeof(double) + 1);
    if (!W || !y) { free(W); if (!y64) free(y); return -1; }
    if (oracle_dequant_awq_bf16_f64(qweight, qzeros, scales, K, N, g, W)) {
        free(W); if (!y64) free(y); return -1;
    }
    const int NB = 256;
    int nblocks = (N + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < nblocks; ++b) {
        int n0 = b * NB, n1 = n0 + NB < N ? n0 + NB : N;
        for (int m = 0; m < M; ++m) {
            double *yr = y + (int64_t)m * N;
            for (int n = n0; n < n1; ++n) yr[n] = 0.0;
            for (int k = 0; k < K; ++k) {
                double xv = oracle_bf16_to_double(x[(int64_t)m * K + k]);
                const double *Wr = W + (int64_t)k * N;
                for (int n = n0; n < n1; ++n) yr[n] += xv * Wr[n];
            }
        }
    }
    if (yb) oracle_double_to_bf16_array(y, (int64_t)M * N, yb);
    free(W);
    if (!y64) free(y);
    return 0;
}
