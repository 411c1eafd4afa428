/*
 * Plain CPU oracle for the block-verification hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the parity reference that the CUDA
 * library is checked against. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg build, load or call it; the product path never
 * does. It shares no code, header, table or helper with the CUDA sources.
 *
 * Everything is scalar C in double precision, written to be read side by side
 * with the definitions it follows:
 *
 *  - The W4 verification projection (dflash-mlx #7 "perf: tune DFlash2 M=8
 *    verification for M1 and M2", PR description: VerifyQuantizedLinear runs
 *    the target's verify block through 4-bit quantized weights). Each weight
 *    is an unsigned 4-bit code with one affine (scale, bias) pair per group of
 *    64 consecutive k:   w(n,k) = scale[n][k/64] * code(n,k) + bias[n][k/64].
 *    Code k of row n sits in bits 4*(k%8) .. 4*(k%8)+3 of word qw[n][k/8]
 *    (eight codes per 32-bit word along K, lowest nibble first).
 *    y[m][n] = sum over k = 0..K-1, in ascending k, of x[m][k] * w(n,k).
 *    All M rows of the block use the same weights (ds4 #778 "dspark: fold
 *    first-token forward into verify ...", commit 1 message: the row tiles
 *    that stop reading every dense weight twice).
 *
 *  - The greedy target token of a verify row is the arg max of its logits
 *    (ds4 #778, commit 1 message: greedy, temperature 0). The decision is
 *    taken on logits rounded to fp32, the precision the GPU path keeps its
 *    accumulators in; ties go to the lowest index; NaN never wins.
 *
 *  - The accept walk (mlxcel #2865 "perf(speculative): commit per-row accepts
 *    in batched DFlash", Summary and commit message): for every batch row, the
 *    length of the longest prefix of drafted tokens equal to the target's
 *    greedy tokens.
 *
 *  - The per-row KV commit (mlxcel #2865, Summary): each row moves its kept
 *    verify-block slots to the end of its own valid prefix, so the cache is
 *    again a contiguous valid prefix per row.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (see oracle/__init__.py). OpenMP, when
 * present, only splits independent output columns n across threads; the order
 * of every sum is the one written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Activation dtype tags, as the test harness passes them. */
enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F32 = 2 };

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);      /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double f32_bits_to_double(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double act_to_double(const void *x, int dtype, size_t i)
{
    if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t *)x)[i]);
    if (dtype == ORACLE_F16) return f16_bits_to_double(((const uint16_t *)x)[i]);
    return f32_bits_to_double(((const uint32_t *)x)[i]);
}

/* The 4-bit code of weight (n, k). */
static unsigned code_at(const uint32_t *qw, int K, int n, int k)
{
    uint32_t word = qw[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
    return (word >> (4 * (k % 8))) & 0xFu;
}

/* Exposed so the tests can pin the bit decoders against library routines. */
double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }
double oracle_f16_to_double(uint16_t h) { return f16_bits_to_double(h); }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * The W4 verification projection.
 *   x      [M][K] activations (bf16, f16 or f32 bits, row-major)
 *   qw     [N][K/8] packed codes, scales / biases [N][K/64] bf16 bits
 *   cols   optional list of n_cols output columns to compute (NULL: all N,
 *          n_cols ignored); y is then [M][n_cols] in list order, else [M][N].
 *   y      fp64 results, unrounded.
 * Returns 0, or -1 on a shape the definition does not cover.
 */
int oracle_vq_linear(const void *x, int act_dtype, int M, int K, int N,
                     const uint32_t *qw, const uint16_t *scales, const uint16_t *biases,
                     const int32_t *cols, int n_cols, double *y, int n_threads)
{
    if (M < 1 || K < 64 || K % 64 != 0 || N < 1) return -1;
    if (act_dtype < ORACLE_BF16 || act_dtype > ORACLE_F32) return -1;
    int n_out = cols ? n_cols : N;
    if (n_out < 0) return -1;

    double *xd = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!xd) return -1;
    for (size_t i = 0; i < (size_t)M * (size_t)K; ++i) xd[i] = act_to_double(x, act_dtype, i);

    int groups = K / 64;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel num_threads(n_threads) reduction(| : bad)
#endif
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
        if (!w) {
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
            for (int j = 0; j < n_out; ++j) {
                int n = cols ? cols[j] : j;
                if (n < 0 || n >= N) { bad = 1; continue; }
                /* dequantize row n: w = scale * code + bias, per 64-wide group */
                for (int k = 0; k < K; ++k) {
                    size_t gi = (size_t)n * (size_t)groups + (size_t)(k / 64);
                    double s = bf16_bits_to_double(scales[gi]);
                    double b = bf16_bits_to_double(biases[gi]);
                    w[k] = s * (double)code_at(qw, K, n, k) + b;
                }
                for (int m = 0; m < M; ++m) {
                    const double *xr = xd + (size_t)m * (size_t)K;
                    double acc = 0.0;
                    for (int k = 0; k < K; ++k) acc += xr[k] * w[k];
                    y[(size_t)m * (size_t)n_out + (size_t)j] = acc;
                }
            }
            free(w);
        }
    }
    free(xd);
    return bad ? -1 : 0;
}

/*
 * Greedy target token per row: arg max over n of logits[m][n] after rounding
 * each logit to fp32. Ties keep the lowest index (strict '>' while scanning n
 * upwards); NaN is skipped; a row with no non-NaN entry gives index 0 and a
 * NaN max. second[m] (optional) is the largest rounded logit at any index
 * other than the winner (-inf if there is none): the margin to the runner-up.
 */
void oracle_argmax(const double *logits, int M, int N, int32_t *idx, float *maxval,
                   float *second)
{
    for (int m = 0; m < M; ++m) {
        const double *row = logits + (size_t)m * (size_t)N;
        int best = -1;
        float bv = 0.0f;
        for (int n = 0; n < N; ++n) {
            float v = (float)row[n];
            if (isnan(v)) continue;
            if (best < 0 || v > bv) { best = n; bv = v; }
        }
        idx[m] = best < 0 ? 0 : best;
        if (maxval) maxval[m] = best < 0 ? NAN : bv;
        if (second) {
            float sv = -INFINITY;
            for (int n = 0; n < N; ++n) {
                float v = (float)row[n];
                if (n == best || isnan(v)) continue;
                if (v > sv) sv = v;
            }
            second[m] = sv;
        }
    }
}

/*
 * Accept walk: accept[b] = number of leading positions j with
 * draft[b][j] == target[b][j] (L when all match).
 */
void oracle_accept_walk(const int32_t *draft, const int32_t *target, int B, int L,
                        int32_t *accept)
{
    for (int b = 0; b < B; ++b) {
        int a = 0;
        while (a < L && draft[(size_t)b * L + a] == target[(size_t)b * L + a]) ++a;
        accept[b] = a;
    }
}

/*
 * Per-row KV commit. Each of the n_tensors tensors is [B][H][S_cap][D] with
 * elements of elem_bytes bytes. For every row b whose numbers are in range,
 * slots src_off[b] .. src_off[b]+keep[b]-1 of every (tensor, b, h) are copied,
 * as they were before the call, to slots prefix_len[b] .. prefix_len[b]+keep[b]-1,
 * and new_len[b] = prefix_len[b] + keep[b]. A row out of range (keep outside
 * 0..max_keep, or either slot range outside 0..S_cap) is left untouched,
 * gets new_len[b] = -1, and sets bit 0 of *status.
 */
void oracle_kv_compact(void **tensors, int n_tensors, int B, int H, int S_cap, int D,
                       int elem_bytes, const int32_t *prefix_len, const int32_t *src_off,
                       const int32_t *keep, int max_keep, int32_t *new_len,
                       int32_t *status)
{
    size_t slot_bytes = (size_t)D * (size_t)elem_bytes;
    unsigned char *tmp = (unsigned char *)malloc(slot_bytes * (size_t)(max_keep > 0 ? max_keep : 1));
    int32_t st = 0;
    for (int b = 0; b < B; ++b) {
        int p = prefix_len[b], s = src_off[b], c = keep[b];
        int ok = c >= 0 && c <= max_keep && p >= 0 && s >= 0 && p + c <= S_cap && s + c <= S_cap;
        if (!ok) {
            new_len[b] = -1;
            st |= 1;
            continue;
        }
        for (int t = 0; t < n_tensors; ++t) {
            unsigned char *base = (unsigned char *)tensors[t];
            for (int h = 0; h < H; ++h) {
                unsigned char *row = base + (((size_t)b * H + h) * (size_t)S_cap) * slot_bytes;
                /* read every kept slot first, then write: source and
                   destination ranges may overlap */
                memcpy(tmp, row + (size_t)s * slot_bytes, (size_t)c * slot_bytes);
                memcpy(row + (size_t)p * slot_bytes, tmp, (size_t)c * slot_bytes);
            }
        }
        new_len[b] = p + c;
    }
    if (status) *status = st;
    free(tmp);
}
