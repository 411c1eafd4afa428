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
 *    read each dense weight once instead of twice).
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

/*
 * Rounding to a 16-bit storage format, to nearest with ties to even.
 *
 * A binary format with `frac` fraction bits and smallest normal exponent emin
 * holds, in the binade [2^e, 2^(e+1)), the multiples of 2^(e - frac); below
 * 2^emin (the subnormals) the multiples of 2^(emin - frac). v / spacing is
 * exact in double (a power-of-two scaling), so rint() (ties to even in the
 * default rounding mode) picks the nearest representable neighbour. A
 * magnitude that rounds above the largest finite value becomes infinite.
 *   binary16: frac 10, emin -14, largest finite 65504
 *   bfloat16: frac 7,  emin -126, largest finite (2 - 2^-7) * 2^127
 */
static double round_to_format(double v, int frac, int emin, double max_finite)
{
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e;
    frexp(fabs(v), &e);            /* |v| = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int lead = e - 1;
    if (lead < emin) lead = emin;
    double spacing = ldexp(1.0, lead - frac);
    double r = rint(v / spacing) * spacing;
    if (fabs(r) > max_finite) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

static double round_to_storage(double v, int dtype)
{
    if (dtype == ORACLE_BF16) return round_to_format(v, 7, -126, ldexp(2.0 - ldexp(1.0, -7), 127));
    return round_to_format(v, 10, -14, 65504.0);
}

/* Bits of a value that is already representable in the storage format. */
static uint16_t storage_bits(double r, int dtype)
{
    if (dtype == ORACLE_BF16) {
        float f = (float)r;                       /* exact: bf16 values are binary32 values */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    uint16_t sign = signbit(r) ? 0x8000u : 0u;
    double a = fabs(r);
    if (isnan(r)) return 0x7E00u;
    if (isinf(r)) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14))                      /* zero or subnormal: a = f * 2^-24 */
        return (uint16_t)(sign | (uint16_t)(a * ldexp(1.0, 24)));
    int e;
    frexp(a, &e);
    int lead = e - 1;                             /* a = (1 + m/1024) * 2^lead */
    uint16_t m = (uint16_t)((ldexp(a, -lead) - 1.0) * 1024.0);
    return (uint16_t)(sign | (uint16_t)((lead + 15) << 10) | m);
}

static double storage_to_double(uint16_t h, int dtype)
{
    return dtype == ORACLE_BF16 ? bf16_bits_to_double(h) : f16_bits_to_double(h);
}

/* Exposed so the tests can pin the rounding against library conversions. */
uint16_t oracle_round_bits(double v, int dtype) { return storage_bits(round_to_storage(v, dtype), dtype); }

/*
 * Rotary position embedding of one head vector at position `pos`, in the
 * half-split pairing: within the first rotary_dim dimensions, dimension i
 * (i < rotary_dim/2) pairs with i + rotary_dim/2, and the pair turns by the
 * angle pos * theta^(-2i / rotary_dim):
 *     y[i]        = x[i] cos a - x[i + h] sin a
 *     y[i + h]    = x[i + h] cos a + x[i] sin a        (h = rotary_dim / 2)
 * Dimensions rotary_dim .. D-1 pass through.
 */
static void rope_vector(const double *x, double *y, int D, int rotary_dim, double pos,
                        double theta)
{
    int h = rotary_dim / 2;
    for (int i = 0; i < h; ++i) {
        double a = pos * pow(theta, -2.0 * (double)i / (double)rotary_dim);
        double c = cos(a), s = sin(a);
        y[i] = x[i] * c - x[i + h] * s;
        y[i + h] = x[i + h] * c + x[i] * s;
    }
    for (int d = rotary_dim; d < D; ++d) y[d] = x[d];
}

/*
 * Verify-block attention over the per-row cache (mlxcel #2865 "perf(speculative):
 * commit per-row accepts in batched DFlash", Summary and commit message: once each
 * row keeps its own accept count, the verify block is rotated and attends at every
 * row's own logical positions, and the stale gap between the row's valid prefix and
 * the shared verify slots is masked for every query).
 *
 * Layouts (16-bit storage, dtype bf16 or f16 for every tensor):
 *   q         [B][L][Hq][D]   the verify block's queries, before rotation
 *   k_new     [B][L][Hkv][D]  its keys, before rotation;  v_new the same for values
 *   k_cache, v_cache [B][Hkv][S_cap][D]: row b holds its valid prefix in slots
 *             0 .. prefix_len[b]-1 (keys stored rotated), and the verify block is
 *             appended at slots src_off[b] .. src_off[b]+L-1.
 * For each row b (P = prefix_len[b], S = src_off[b]) and block position j:
 *   1. the logical position of the block's token j is P + j; its key is rotated
 *      there, rounded to the storage format and written to slot S + j of k_cache,
 *      and its value is copied to slot S + j of v_cache;
 *   2. its query (head hq, kv head hq / (Hq / Hkv)) is rotated at P + j and rounded
 *      to the storage format;
 *   3. it attends, with softmax(scale * q.k), to the cache slots 0 .. P-1 and to the
 *      block's slots S .. S + j (causal within the block); slots P .. S-1, the stale
 *      gap, and everything after S + j are masked out.
 * out      [B][L][Hq][D] fp64, unrounded.
 * k_rot    optional [B][L][Hkv][D] fp64: the rotated keys before rounding.
 * A row with P < 0, S < P or S + L > S_cap is left untouched in the caches, gets
 * zero outputs, and sets bit 0 of *status (status optional).
 * Returns 0, or -1 on a shape the definition does not cover.
 */
int oracle_verify_attention(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                            uint16_t *k_cache, uint16_t *v_cache, const int32_t *prefix_len,
                            const int32_t *src_off, int B, int L, int Hq, int Hkv, int D,
                            int S_cap, int rotary_dim, double theta, double scale, int dtype,
                            double *out, double *k_rot, int32_t *status, int n_threads)
{
    if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || S_cap < L) return -1;
    if (rotary_dim < 0 || rotary_dim > D || rotary_dim % 2 != 0) return -1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    const int G = Hq / Hkv;
    int32_t st = 0;
    memset(out, 0, sizeof(double) * (size_t)B * L * Hq * D);
    if (k_rot) memset(k_rot, 0, sizeof(double) * (size_t)B * L * Hkv * D);

    double *xv = (double *)malloc(sizeof(double) * (size_t)D);
    double *yv = (double *)malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b], S = src_off[b];
        if (P < 0 || S < P || S + L > S_cap) {
            st |= 1;
            continue;
        }
        /* step 1: the block's keys and values go to slots S .. S+L-1 */
        for (int j = 0; j < L; ++j)
            for (int h = 0; h < Hkv; ++h) {
                size_t src = (((size_t)b * L + j) * Hkv + h) * D;
                size_t dst = (((size_t)b * Hkv + h) * S_cap + (size_t)(S + j)) * D;
                for (int d = 0; d < D; ++d) xv[d] = storage_to_double(k_new[src + d], dtype);
                rope_vector(xv, yv, D, rotary_dim, (double)(P + j), theta);
                for (int d = 0; d < D; ++d) {
                    if (k_rot) k_rot[src + d] = yv[d];
                    k_cache[dst + d] = storage_bits(round_to_storage(yv[d], dtype), dtype);
                    v_cache[dst + d] = v_new[src + d];
                }
            }
    }
    free(xv);
    free(yv);

    /* steps 2 and 3, one query (b, j, hq) at a time */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic) num_threads(n_threads > 0 ? n_threads : 1)
#endif
    for (long long qi = 0; qi < (long long)B * L * Hq; ++qi) {
        int hq = (int)(qi % Hq);
        int j = (int)((qi / Hq) % L);
        int b = (int)(qi / ((long long)Hq * L));
        int P = prefix_len[b], S = src_off[b];
        if (P < 0 || S < P || S + L > S_cap) continue;
        int hk = hq / G;
        int n_vis = P + j + 1;
        double *qv = (double *)malloc(sizeof(double) * (size_t)D * 2);
        double *sc = (double *)malloc(sizeof(double) * (size_t)n_vis);
        size_t qoff = (size_t)qi * D;     /* [B][L][Hq][D] flattened in the same order */
        for (int d = 0; d < D; ++d) qv[D + d] = storage_to_double(q[qoff + d], dtype);
        rope_vector(qv + D, qv, D, rotary_dim, (double)(P + j), theta);
        for (int d = 0; d < D; ++d) qv[d] = round_to_storage(qv[d], dtype);

        const uint16_t *kb = k_cache + ((size_t)b * Hkv + hk) * (size_t)S_cap * D;
        const uint16_t *vb = v_cache + ((size_t)b * Hkv + hk) * (size_t)S_cap * D;
        /* visible slot number t: the prefix slot t for t < P, else the block slot S + (t - P) */
        double mx = -INFINITY;
        for (int t = 0; t < n_vis; ++t) {
            size_t slot = (size_t)(t < P ? t : S + (t - P));
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qv[d] * storage_to_double(kb[slot * D + d], dtype);
            sc[t] = scale * dot;
            if (sc[t] > mx) mx = sc[t];
        }
        double l = 0.0;
        for (int t = 0; t < n_vis; ++t) {
            sc[t] = exp(sc[t] - mx);
            l += sc[t];
        }
        double *o = out + qoff;
        for (int t = 0; t < n_vis; ++t) {
            size_t slot = (size_t)(t < P ? t : S + (t - P));
            for (int d = 0; d < D; ++d) o[d] += sc[t] * storage_to_double(vb[slot * D + d], dtype);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
        free(qv);
        free(sc);
    }
    if (status) *status = st;
    return 0;
}
