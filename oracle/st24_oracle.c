/*
 * st24_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU oracle for 2:4 structured sparsity:
 * magnitude prune, compress to (kept values, 2-bit in-group indices),
 * decompress, and the sparse x dense product C = alpha*(A_sparse*B) + beta*C.
 * Floating-point arithmetic is fp64; int8 products are summed in int64.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline use this file.  The CUDA library never links, includes or calls
 * it, and this file includes nothing from the library.
 *
 * Sources (web pages, cited by title and section):
 *  [CH26] "Chapter 26 -- Sparsity: The Hardware View":
 *     - section "2:4 Fine-Grained Structured Sparsity": in every contiguous
 *       group of 4 weights exactly 2 are zero; the worked example (dense row
 *       w0..w7 -> pruned [w0 0 0 w3 | 0 w5 w6 0] -> values [w0 w3 | w5 w6],
 *       indices [0 3 | 1 2], 2 bits per kept value, 4 bits per group); the
 *       stored pair is multiplied against the 2 activations its indices
 *       select, the other 2 products being zero.
 *     - section "Python: Build a 2:4 Mask, Compress It, and Show Why
 *       Unstructured Doesn't Help": the mask keeps the 2 largest-|w| of each
 *       group of 4 along the last dimension (K divisible by 4); compression
 *       keeps those 2 positions sorted ascending and gathers their values.
 *  [SS24] "10.4g Structured Sparsity (2:4)", section "What is 2:4 Structured
 *       Sparsity?": 2 non-zero of every 4 consecutive values.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *  R1 ties: the pages rank by |w| with an argsort that does not promise a
 *     stable order.  Here the kept pair is the 2 largest |w| with ties going
 *     to the LOWER index (first the largest, earliest on a tie; then the
 *     largest of the other three, earliest on a tie).
 *  R2 magnitude is |w| of the decoded real value; +0 and -0 are equal.  A NaN
 *     ranks above every number (so it is kept), and NaNs tie with each other.
 *  R3 exactly 2 slots are kept per group even when the group has fewer than 2
 *     non-zeros; the dropped slots are +0 (all-zero bits) of the type.
 *  R4 metadata bit order (the pages say only "2 bits each"): group g of a row
 *     is the nibble (i0 | i1 << 2) with i0 < i1, packed two groups per byte
 *     along K, group g in bits 4*(g%2) of byte g/2.  A row of K elements has
 *     ceil(K/8) metadata bytes.
 *  R5 values are row-major M x K/2 in the element type, the pair of group g
 *     at columns 2g (index i0) and 2g+1 (index i1).
 *  R6 the product sums k in ascending order; beta == 0 means C is not read.
 *  R7 the per-row quantisation before the prune (see orc_quantize_prune_compress).
 *  R8 N:M pruning written in the 2:4 form (see orc_prune_compress_nm).
 *  R9 the transposed product sums m in ascending order (see orc_spmm_t).
 *  R10 N:M pruning with up to four kept per 4-subgroup written as two 2:4
 *     forms whose sum is the pruned matrix (see orc_prune_compress_nm2).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Element types the oracle understands (its own numbering). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_S8 = 3, ORC_F32 = 4, ORC_S32 = 5 };

static int elem_size(int dt)
{
    switch (dt) {
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_E4M3: case ORC_S8: return 1;
    case ORC_F32: case ORC_S32: return 4;
    default: return 0;
    }
}

int orc_elem_size(int dt) { return elem_size(dt); }

/* ---------------------------------------------------------------- decoding */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
static double dec_f16(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double dec_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite 448. */
static double dec_e4m3(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 0xf, m = b & 7;
    double v;
    if (e == 0) v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
    else if (e == 15 && m == 7) v = NAN;
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

static double dec_f32(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Value of element i of a typed buffer, as a double. */
static double load_real(int dt, const void* p, int64_t i)
{
    switch (dt) {
    case ORC_F16: return dec_f16(((const uint16_t*)p)[i]);
    case ORC_BF16: return dec_bf16(((const uint16_t*)p)[i]);
    case ORC_E4M3: return dec_e4m3(((const uint8_t*)p)[i]);
    case ORC_S8: return (double)((const int8_t*)p)[i];
    case ORC_F32: return dec_f32(((const uint32_t*)p)[i]);
    case ORC_S32: return (double)((const int32_t*)p)[i];
    default: return NAN;
    }
}

void orc_decode(int dt, const void* in, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = load_real(dt, in, i);
}

/* ------------------------------------------------------- prune (selection) */

/* |a| > |b| in the order of reading R2 (NaN above every number). */
static int mag_greater(double a, double b)
{
    int na = isnan(a), nb = isnan(b);
    if (na || nb) return na && !nb;
    return fabs(a) > fabs(b);
}

/* The kept pair of one group of 4 values (reading R1), returned ascending. */
static void select_pair(const double v[4], int* i0, int* i1)
{
    int first = 0;
    for (int j = 1; j < 4; ++j)
        if (mag_greater(v[j], v[first])) first = j;        /* strict: earlier index wins a tie */
    int second = (first == 0) ? 1 : 0;
    for (int j = 0; j < 4; ++j)
        if (j != first && mag_greater(v[j], v[second])) second = j;
    *i0 = first < second ? first : second;
    *i1 = first < second ? second : first;
}

int64_t orc_meta_row_bytes(int64_t K) { return (K / 4 + 1) / 2; }

/* Closed-form storage of the compressed form (values + metadata), in bytes. */
int64_t orc_values_bytes(int dt, int64_t M, int64_t K) { return M * (K / 2) * elem_size(dt); }
int64_t orc_meta_bytes(int64_t M, int64_t K) { return M * orc_meta_row_bytes(K); }

/*
 * Prune W (M x K, row stride ldw elements) and write, for every row and group:
 *   pruned (M x K, row stride K, may be NULL): W with the two dropped slots set to +0,
 *   mask   (M x K bytes, may be NULL): 1 where kept, 0 where dropped,
 *   values (M x K/2, may be NULL) and meta (M x ceil(K/8) bytes, may be NULL):
 *          the compressed form of readings R4 and R5.
 * Returns 0, or -1 if K is not a multiple of 4 or the type is unknown.
 */
int orc_prune_compress(int dt, const void* W, int64_t M, int64_t K, int64_t ldw,
                       void* pruned, uint8_t* mask, void* values, uint8_t* meta)
{
    int es = elem_size(dt);
    if (K % 4 != 0 || es == 0 || dt == ORC_S32) return -1;
    const uint8_t* w = (const uint8_t*)W;
    int64_t mrb = orc_meta_row_bytes(K);
    if (meta) memset(meta, 0, (size_t)(M * mrb));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < K / 4; ++g) {
            double v[4];
            for (int j = 0; j < 4; ++j) v[j] = load_real(dt, w + (m * ldw) * es, 4 * g + j);
            int i0, i1;
            select_pair(v, &i0, &i1);
            for (int j = 0; j < 4; ++j) {
                int keep = (j == i0 || j == i1);
                const uint8_t* src = w + (m * ldw + 4 * g + j) * es;
                if (pruned) {
                    uint8_t* dst = (uint8_t*)pruned + (m * K + 4 * g + j) * es;
                    if (keep) memcpy(dst, src, es);
                    else memset(dst, 0, es);
                }
                if (mask) mask[m * K + 4 * g + j] = (uint8_t)keep;
            }
            if (values) {
                uint8_t* vrow = (uint8_t*)values + (m * (K / 2)) * es;
                memcpy(vrow + (2 * g) * es, w + (m * ldw + 4 * g + i0) * es, es);
                memcpy(vrow + (2 * g + 1) * es, w + (m * ldw + 4 * g + i1) * es, es);
            }
            if (meta) {
                uint8_t nib = (uint8_t)(i0 | (i1 << 2));
                meta[m * mrb + g / 2] |= (uint8_t)(nib << (4 * (g % 2)));
            }
        }
    }
    return 0;
}

/* ------------------------------------- quantise, then prune and compress */

/*
 * fp32 -> OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * normal values (1 + m/8) * 2^(e-7), subnormals m/8 * 2^-6, largest finite
 * 448), rounding to nearest with ties to even, magnitudes at or above 448
 * saturated to 448.  x must be finite.
 */
static uint8_t enc_e4m3_sat(float x)
{
    uint8_t s = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);                /* exact */
    if (a >= 448.0) return s | 0x7E;           /* 1.1111.110 = 448 */
    if (a == 0.0) return s;
    int e;
    (void)frexp(a, &e);                        /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < -6) {
        /* subnormal binade: units of 2^-9; 8 units is the smallest normal */
        double q = nearbyint(ldexp(a, 9));
        return s | (uint8_t)q;
    }
    double q = nearbyint(ldexp(a, 3 - E));     /* the significand in eighths: 8..16 */
    int mant = (int)q - 8;
    if (mant == 8) { E += 1; mant = 0; }
    int code = ((E + 7) << 3) | mant;
    if (code > 0x7E) code = 0x7E;
    return s | (uint8_t)code;
}

/* fp32 -> int8 rounding to nearest with ties to even, clamped to [-127, 127]. */
static int8_t enc_s8_sat(float x)
{
    float r = nearbyintf(x);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int8_t)r;
}

uint8_t orc_enc_e4m3(float x) { return enc_e4m3_sat(x); }

/*
 * Per-row quantisation of a 16-bit weight followed by the prune and compress
 * above ("Chapter 26 -- Sparsity: The Hardware View", section "Sparsity +
 * Quantization Combine": 2:4 sparsity and 8-bit weights stack; "Establishing
 * a Scalable Sparse Ecosystem with the Universal Sparse Tensor Abstraction",
 * section "Building a Practical Compression Pipeline": prune plus INT8
 * post-training quantisation).  The pages give the pipeline, not its
 * arithmetic; reading R7:
 *   amax  = max |w| over the row (w decoded exactly to fp32);
 *   inv   = Q / amax in fp32 (Q = 448 for e4m3, 127 for int8);
 *   code  = encode(fp32(w) * inv), the product rounded once to fp32, then
 *           encoded as above (e4m3: nearest-even, saturated; int8: nearest-
 *           even, clamped to [-127, 127]);
 *   scale = amax / Q in fp32, so that w ~ code * scale;
 *   a row with amax = 0 gets scale 0 and all-zero codes.
 * The codes of the row are then pruned and compressed exactly as by
 * orc_prune_compress (the dst type's magnitude order).  W must be finite.
 * codes (M x K, may be NULL) receives the quantised rows before pruning.
 * Returns 0, or -1 for an unknown type pair or K not a multiple of 4.
 */
int orc_quantize_prune_compress(int src, int dst, const void* W, int64_t M, int64_t K, int64_t ldw,
                                void* codes, void* values, uint8_t* meta, float* scales)
{
    if ((src != ORC_F16 && src != ORC_BF16) || (dst != ORC_E4M3 && dst != ORC_S8) || K % 4 != 0) return -1;
    const float Q = dst == ORC_E4M3 ? 448.0f : 127.0f;
    uint8_t* row = (uint8_t*)malloc((size_t)(K > 0 ? K : 1));
    if (!row) return -1;
    int64_t mrb = orc_meta_row_bytes(K);
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* wr = (const uint16_t*)W + m * ldw;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = (float)fabs(load_real(src, wr, k));
            if (a > amax) amax = a;
        }
        float inv = amax > 0.0f ? Q / amax : 0.0f;
        scales[m] = amax > 0.0f ? amax / Q : 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float y = (float)load_real(src, wr, k) * inv;
            row[k] = dst == ORC_E4M3 ? enc_e4m3_sat(y) : (uint8_t)enc_s8_sat(y);
        }
        if (codes) memcpy((uint8_t*)codes + m * K, row, (size_t)K);
        int rc = orc_prune_compress(dst, row, 1, K, K, NULL, NULL,
                                    values ? (uint8_t*)values + m * (K / 2) : NULL,
                                    meta ? meta + m * mrb : NULL);
        if (rc != 0) { free(row); return rc; }
    }
    free(row);
    return 0;
}

/* ------------------------------------------- N:M prune into the 2:4 form */

/*
 * N:M generalisations ("Chapter 26 -- Sparsity: The Hardware View", section
 * "Block Sparsity, N:M Generalizations, and Channel Pruning": 1:4, 2:8 and
 * friends keep N of every M consecutive weights).  Reading R8: in every group
 * of M consecutive elements along K keep the N of largest magnitude, ties to
 * the lower index (the order of reading R2), chosen one at a time like
 * select_pair.  With M = 4 or 8 and N <= 2 every aligned 4-element subgroup
 * keeps at most 2 elements, so the result is written in the 2:4 compressed
 * form: a subgroup with 2 kept elements stores them; with 1, the kept one
 * and the lowest-index dropped one as a +0 partner; with none, indices 0
 * and 1 with +0 values.  The pair is stored in ascending index order.
 * pruned (M x K, may be NULL) receives W with every dropped element +0.
 * Returns 0, or -1 for an unsupported (n, m), a K not a multiple of m or an
 * unknown type.
 */
int orc_prune_compress_nm(int dt, int n, int m, const void* W, int64_t M, int64_t K, int64_t ldw,
                          void* pruned, void* values, uint8_t* meta)
{
    int es = elem_size(dt);
    if (es == 0 || dt == ORC_S32 || dt == ORC_F32 || (m != 4 && m != 8) || n < 1 || n > 2 || K % m != 0) return -1;
    const uint8_t* w = (const uint8_t*)W;
    int64_t mrb = orc_meta_row_bytes(K);
    if (meta) memset(meta, 0, (size_t)(M * mrb));
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t g0 = 0; g0 < K; g0 += m) {
            double v[8];
            int keep[8] = {0};
            for (int j = 0; j < m; ++j) v[j] = load_real(dt, w + (r * ldw) * es, g0 + j);
            for (int t = 0; t < n; ++t) {           /* the t-th largest: first maximum not yet kept */
                int best = -1;
                for (int j = 0; j < m; ++j)
                    if (!keep[j] && (best < 0 || mag_greater(v[j], v[best]))) best = j;
                keep[best] = 1;
            }
            for (int j = 0; j < m; ++j) {
                if (!pruned) continue;
                uint8_t* dst = (uint8_t*)pruned + (r * K + g0 + j) * es;
                if (keep[j]) memcpy(dst, w + (r * ldw + g0 + j) * es, es);
                else memset(dst, 0, es);
            }
            for (int q = 0; q < m / 4; ++q) {       /* the 4-element subgroups, in the 2:4 form */
                int idx[2], cnt = 0;
                for (int j = 0; j < 4 && cnt < 2; ++j)
                    if (keep[4 * q + j]) idx[cnt++] = j;
                int nk = cnt;
                for (int j = 0; j < 4 && cnt < 2; ++j)    /* fill with the lowest dropped indices */
                    if (!keep[4 * q + j] && (cnt == 0 || j != idx[0])) idx[cnt++] = j;
                int i0 = idx[0] < idx[1] ? idx[0] : idx[1], i1 = idx[0] < idx[1] ? idx[1] : idx[0];
                int64_t g = (g0 + 4 * q) / 4;
                if (values) {
                    uint8_t* vrow = (uint8_t*)values + (r * (K / 2)) * es;
                    const int ii[2] = {i0, i1};
                    for (int h = 0; h < 2; ++h) {
                        uint8_t* dst = vrow + (2 * g + h) * es;
                        if (keep[4 * q + ii[h]]) memcpy(dst, w + (r * ldw + 4 * g + ii[h]) * es, es);
                        else memset(dst, 0, es);
                    }
                }
                (void)nk;
                if (meta) meta[r * mrb + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
            }
        }
    }
    return 0;
}

/*
 * N:M pruning with up to four kept elements per aligned 4-element subgroup
 * (4:8, 3:8, ...; "Chapter 26 -- Sparsity: The Hardware View", section "Block
 * Sparsity, N:M Generalizations, and Channel Pruning").  Reading R10: keep the
 * n largest |w| of every m consecutive elements along K exactly as
 * orc_prune_compress_nm does (chosen one at a time, ties to the lower index),
 * then write the result as TWO 2:4 compressed forms whose sum is the pruned
 * matrix: in every 4-element subgroup the kept elements in ascending index
 * order go first to form 0 (its first two) and then to form 1 (the rest); a
 * form holding fewer than two of the subgroup's elements takes as the missing
 * slots the lowest indices of the subgroup not among its own, with +0 values.
 * The forms are stored concatenated along K, so that together they are the
 * 2:4 form of an M x 2K matrix [form 0 | form 1]:
 *   values (M x K): row r = form 0's K/2 values, then form 1's K/2 values;
 *   meta   (M x 2*ceil(K/8) bytes): row r = form 0's ceil(K/8) bytes, then form 1's.
 * Multiplying that M x 2K matrix by B stacked twice ([B; B], 2K x N) gives the
 * pruned matrix times B.  pruned (M x K, may be NULL) receives W with every
 * dropped element +0.  Supported: m in {4, 8}, 1 <= n <= min(4, m), K % m == 0.
 * Returns 0, or -1 for unsupported arguments.
 */
int orc_prune_compress_nm2(int dt, int n, int m, const void* W, int64_t M, int64_t K, int64_t ldw,
                           void* pruned, void* values, uint8_t* meta)
{
    int es = elem_size(dt);
    if (es == 0 || dt == ORC_S32 || dt == ORC_F32 || (m != 4 && m != 8) || n < 1 || n > 4 || n > m || K % m != 0)
        return -1;
    const uint8_t* w = (const uint8_t*)W;
    int64_t mrb = orc_meta_row_bytes(K);
    if (meta) memset(meta, 0, (size_t)(M * 2 * mrb));
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t g0 = 0; g0 < K; g0 += m) {
            double v[8];
            int keep[8] = {0};
            for (int j = 0; j < m; ++j) v[j] = load_real(dt, w + (r * ldw) * es, g0 + j);
            for (int t = 0; t < n; ++t) {           /* the t-th largest: first maximum not yet kept */
                int best = -1;
                for (int j = 0; j < m; ++j)
                    if (!keep[j] && (best < 0 || mag_greater(v[j], v[best]))) best = j;
                keep[best] = 1;
            }
            for (int j = 0; j < m; ++j) {
                if (!pruned) continue;
                uint8_t* dst = (uint8_t*)pruned + (r * K + g0 + j) * es;
                if (keep[j]) memcpy(dst, w + (r * ldw + g0 + j) * es, es);
                else memset(dst, 0, es);
            }
            for (int q = 0; q < m / 4; ++q) {
                int kept[4], nk = 0;
                for (int j = 0; j < 4; ++j)
                    if (keep[4 * q + j]) kept[nk++] = j;
                int64_t g = (g0 + 4 * q) / 4;
                for (int f = 0; f < 2; ++f) {
                    int own[2], no = 0;                 /* this form's kept elements of the subgroup */
                    for (int t = 2 * f; t < nk && t < 2 * f + 2; ++t) own[no++] = kept[t];
                    int idx[2], isval[2], c = 0;
                    for (int t = 0; t < no; ++t) { idx[c] = own[t]; isval[c] = 1; ++c; }
                    for (int j = 0; j < 4 && c < 2; ++j) {   /* lowest indices not among its own */
                        int mine = 0;
                        for (int t = 0; t < no; ++t) mine |= (own[t] == j);
                        if (!mine && (c == 0 || idx[0] != j)) { idx[c] = j; isval[c] = 0; ++c; }
                    }
                    int lo = idx[0] < idx[1] ? 0 : 1;   /* the pair in ascending index order */
                    int i0 = idx[lo], i1 = idx[1 - lo];
                    int v0 = isval[lo], v1 = isval[1 - lo];
                    if (values) {
                        uint8_t* vrow = (uint8_t*)values + (r * K + (int64_t)f * (K / 2)) * es;
                        if (v0) memcpy(vrow + (2 * g) * es, w + (r * ldw + 4 * g + i0) * es, es);
                        else memset(vrow + (2 * g) * es, 0, es);
                        if (v1) memcpy(vrow + (2 * g + 1) * es, w + (r * ldw + 4 * g + i1) * es, es);
                        else memset(vrow + (2 * g + 1) * es, 0, es);
                    }
                    if (meta) meta[r * 2 * mrb + f * mrb + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g % 2)));
                }
            }
        }
    }
    return 0;
}

/* The two indices of group g of row m (reading R4). */
static void meta_pair(const uint8_t* meta, int64_t mrb, int64_t m, int64_t g, int* i0, int* i1)
{
    uint8_t nib = (meta[m * mrb + g / 2] >> (4 * (g % 2))) & 0xf;
    *i0 = nib & 3;
    *i1 = nib >> 2;
}

/*
 * Inverse of compression: scatter the two values of every group to their
 * indices and fill the rest with +0.  W_out is M x K with row stride ldw.
 * Returns 0, -1 on bad arguments, -2 if some group's indices are not
 * strictly ascending (such metadata is not a valid compressed form).
 */
int orc_decompress(int dt, const void* values, const uint8_t* meta, int64_t M, int64_t K,
                   void* W_out, int64_t ldw)
{
    int es = elem_size(dt);
    if (K % 4 != 0 || es == 0) return -1;
    int64_t mrb = orc_meta_row_bytes(K);
    int bad = 0;
    for (int64_t m = 0; m < M; ++m) {
        uint8_t* row = (uint8_t*)W_out + (m * ldw) * es;
        memset(row, 0, (size_t)(K * es));
        for (int64_t g = 0; g < K / 4; ++g) {
            int i0, i1;
            meta_pair(meta, mrb, m, g, &i0, &i1);
            if (!(i0 < i1)) bad = 1;
            const uint8_t* v = (const uint8_t*)values + (m * (K / 2) + 2 * g) * es;
            memcpy(row + (4 * g + i0) * es, v, es);
            memcpy(row + (4 * g + i1) * es, v + es, es);
        }
    }
    return bad ? -2 : 0;
}

/* ---------------------------------------------------------------- products */

/*
 * Sparse x dense product in the compressed form.  A is (values, meta) of an
 * M x K matrix; B is K x N stored with element (k, n) at B[n*ldb + k];
 * C_in and out are M x N with element (m, n) at [n*ldc + m] (out uses ldc=M).
 *   acc(m, n) = sum over groups g ascending, j = 0, 1:
 *               values[m, 2g+j] * B[4g + i_j, n]          (fp64, or int64 for int8)
 *   out(m, n) = alpha * scale[m] * acc + beta * C_in(m, n)  (fp64; scale NULL = 1,
 *               C_in not read when beta == 0)
 * The acc of int8 inputs is also written to acc_i64 (may be NULL).
 */
typedef struct {
    int dt_ab, dt_c;
    int64_t M, N, K, ldb, ldc;
    double alpha, beta;
    const void *values, *B, *C_in;
    const uint8_t* meta;
    const float* scale;
    double* out;
    int64_t* acc_i64;
    /* dense variant */
    const void* A;
    int64_t lda;
    /* sampled variant */
    const int64_t *rows, *cols;
    int64_t nsamples;
    /* work split */
    int64_t begin, end;
} job_t;

/* ------------------------------------------- transposed use (dX = dY * W) */

/*
 * The transposed product of a compressed weight ("Chapter 26 -- Sparsity:
 * The Hardware View", section "2:4: ~2x on the Matmul, Less End-to-End":
 * train dense, prune to 2:4, retrain -- retraining needs the input gradient
 * dX = dY * W of a layer Y = X * W^T).  For A (M x K) in the compressed form,
 *   out(k, n) = alpha * sum over m ascending of A(m, k) * B(m, n)
 *               + beta * C_in(k, n)        (fp64; int64 sums for int8),
 * where A(m, k) is the stored value whose in-group index names k (the first
 * of the pair if i0 names it, the second if i1 does), else 0; B(m, n) is at
 * B[n*ldb + m] (a row-major dY[N, M]); C_in(k, n) and out(k, n) are at
 * [n*ldc + k] and out[n*K + k] (row-major dX[N, K]).  The sum runs along M,
 * along which the weight has no 2:4 structure.
 */
static void a_elem(const job_t* j, int64_t m, int64_t k, double* af, int64_t* ai)
{
    int64_t mrb = (j->K / 4 + 1) / 2;
    int64_t g = k / 4;
    int p = (int)(k % 4);
    uint8_t nib = (j->meta[m * mrb + g / 2] >> (4 * (g % 2))) & 0xf;
    int i0 = nib & 3, i1 = nib >> 2;
    int64_t idx = -1;
    if (p == i0) idx = m * (j->K / 2) + 2 * g;
    else if (p == i1) idx = m * (j->K / 2) + 2 * g + 1;
    if (idx < 0) { *af = 0.0; *ai = 0; return; }
    if (j->dt_ab == ORC_S8) { *ai = ((const int8_t*)j->values)[idx]; *af = (double)*ai; }
    else { *af = load_real(j->dt_ab, j->values, idx); *ai = 0; }
}

static double transposed_elem(const job_t* j, int64_t k, int64_t n, int64_t* acc_i)
{
    double sf = 0.0;
    int64_t si = 0;
    for (int64_t m = 0; m < j->M; ++m) {
        double af;
        int64_t ai;
        a_elem(j, m, k, &af, &ai);
        if (j->dt_ab == ORC_S8) si += ai * (int64_t)((const int8_t*)j->B)[n * j->ldb + m];
        else sf += af * load_real(j->dt_ab, j->B, n * j->ldb + m);
    }
    *acc_i = si;
    double acc = (j->dt_ab == ORC_S8) ? (double)si : sf;
    double r = j->alpha * acc;
    if (j->beta != 0.0) r += j->beta * load_real(j->dt_c, j->C_in, n * j->ldc + k);
    return r;
}

static void* run_rows_t(void* arg)
{
    job_t* j = (job_t*)arg;
    for (int64_t k = j->begin; k < j->end; ++k)
        for (int64_t n = 0; n < j->N; ++n) {
            int64_t ai;
            j->out[n * j->K + k] = transposed_elem(j, k, n, &ai);
            if (j->acc_i64) j->acc_i64[n * j->K + k] = ai;
        }
    return NULL;
}

static void* run_samples_t(void* arg)
{
    job_t* j = (job_t*)arg;
    for (int64_t s = j->begin; s < j->end; ++s) {
        int64_t ai;
        j->out[s] = transposed_elem(j, j->rows[s], j->cols[s], &ai);
        if (j->acc_i64) j->acc_i64[s] = ai;
    }
    return NULL;
}

static double epilogue(const job_t* j, int64_t m, int64_t n, double acc)
{
    double s = j->scale ? (double)j->scale[m] : 1.0;
    double r = j->alpha * s * acc;
    if (j->beta != 0.0) r += j->beta * load_real(j->dt_c, j->C_in, n * j->ldc + m);
    return r;
}

/* One output element from the compressed form. */
static void sparse_dot(const job_t* j, int64_t m, int64_t n, double* acc_f, int64_t* acc_i)
{
    int64_t mrb = orc_meta_row_bytes(j->K);
    double sf = 0.0;
    int64_t si = 0;
    for (int64_t g = 0; g < j->K / 4; ++g) {
        int idx[2];
        meta_pair(j->meta, mrb, m, g, &idx[0], &idx[1]);
        for (int t = 0; t < 2; ++t) {
            int64_t k = 4 * g + idx[t];
            if (j->dt_ab == ORC_S8) {
                int64_t a = ((const int8_t*)j->values)[m * (j->K / 2) + 2 * g + t];
                int64_t b = ((const int8_t*)j->B)[n * j->ldb + k];
                si += a * b;
            } else {
                double a = load_real(j->dt_ab, j->values, m * (j->K / 2) + 2 * g + t);
                double b = load_real(j->dt_ab, j->B, n * j->ldb + k);
                sf += a * b;
            }
        }
    }
    *acc_f = (j->dt_ab == ORC_S8) ? (double)si : sf;
    *acc_i = si;
}

/* One output element from a dense (already pruned) A, plain triple loop. */
static void dense_dot(const job_t* j, int64_t m, int64_t n, double* acc_f, int64_t* acc_i)
{
    double sf = 0.0;
    int64_t si = 0;
    for (int64_t k = 0; k < j->K; ++k) {
        if (j->dt_ab == ORC_S8) {
            si += (int64_t)((const int8_t*)j->A)[m * j->lda + k] * ((const int8_t*)j->B)[n * j->ldb + k];
        } else {
            sf += load_real(j->dt_ab, j->A, m * j->lda + k) * load_real(j->dt_ab, j->B, n * j->ldb + k);
        }
    }
    *acc_f = (j->dt_ab == ORC_S8) ? (double)si : sf;
    *acc_i = si;
}

static void* run_rows(void* arg)
{
    job_t* j = (job_t*)arg;
    for (int64_t m = j->begin; m < j->end; ++m)
        for (int64_t n = 0; n < j->N; ++n) {
            double af;
            int64_t ai;
            if (j->A) dense_dot(j, m, n, &af, &ai);
            else sparse_dot(j, m, n, &af, &ai);
            j->out[n * j->M + m] = epilogue(j, m, n, af);
            if (j->acc_i64) j->acc_i64[n * j->M + m] = ai;
        }
    return NULL;
}

static void* run_samples(void* arg)
{
    job_t* j = (job_t*)arg;
    for (int64_t s = j->begin; s < j->end; ++s) {
        double af;
        int64_t ai;
        int64_t m = j->rows[s], n = j->cols[s];
        sparse_dot(j, m, n, &af, &ai);
        j->out[s] = epilogue(j, m, n, af);
        if (j->acc_i64) j->acc_i64[s] = ai;
    }
    return NULL;
}

static int thread_count(int requested)
{
    if (requested > 0) return requested;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Split [0, total) over threads and run fn on each part; returns threads used. */
static int parallel_for(job_t* base, int64_t total, int nthreads, void* (*fn)(void*))
{
    int nt = thread_count(nthreads);
    if (nt > total) nt = total > 0 ? (int)total : 1;
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * nt);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
    for (int t = 0; t < nt; ++t) {
        jobs[t] = *base;
        jobs[t].begin = total * t / nt;
        jobs[t].end = total * (t + 1) / nt;
        pthread_create(&th[t], NULL, fn, &jobs[t]);
    }
    for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
    return nt;
}

static int check_types(int dt_ab, int dt_c)
{
    if (dt_ab != ORC_F16 && dt_ab != ORC_BF16 && dt_ab != ORC_E4M3 && dt_ab != ORC_S8 && dt_ab != ORC_F32)
        return -1;
    if (elem_size(dt_c) == 0) return -1;
    return 0;
}

/* Full product from the compressed form; out and acc_i64 are N*M, (m, n) at [n*M + m].
 * Returns the number of threads used, or -1 on bad arguments. */
int orc_spmm(int dt_ab, int dt_c, int64_t M, int64_t N, int64_t K, double alpha,
             const void* values, const uint8_t* meta, const void* B, int64_t ldb,
             double beta, const void* C_in, int64_t ldc, const float* scale,
             double* out, int64_t* acc_i64, int nthreads)
{
    if (K % 4 != 0 || check_types(dt_ab, dt_c)) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dt_ab = dt_ab; j.dt_c = dt_c; j.M = M; j.N = N; j.K = K; j.ldb = ldb; j.ldc = ldc;
    j.alpha = alpha; j.beta = beta; j.values = values; j.meta = meta; j.B = B; j.C_in = C_in;
    j.scale = scale; j.out = out; j.acc_i64 = acc_i64;
    return parallel_for(&j, M, nthreads, run_rows);
}

/* The same product from a dense (pruned) A, M x K with row stride lda. */
int orc_gemm_dense(int dt_ab, int dt_c, int64_t M, int64_t N, int64_t K, double alpha,
                   const void* A, int64_t lda, const void* B, int64_t ldb,
                   double beta, const void* C_in, int64_t ldc, const float* scale,
                   double* out, int64_t* acc_i64, int nthreads)
{
    if (check_types(dt_ab, dt_c)) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dt_ab = dt_ab; j.dt_c = dt_c; j.M = M; j.N = N; j.K = K; j.ldb = ldb; j.ldc = ldc;
    j.alpha = alpha; j.beta = beta; j.A = A; j.lda = lda; j.B = B; j.C_in = C_in;
    j.scale = scale; j.out = out; j.acc_i64 = acc_i64;
    return parallel_for(&j, M, nthreads, run_rows);
}

/* Selected outputs (rows[s], cols[s]) of the compressed-form product; out[s]. */
int orc_spmm_sampled(int dt_ab, int dt_c, int64_t M, int64_t N, int64_t K, double alpha,
                     const void* values, const uint8_t* meta, const void* B, int64_t ldb,
                     double beta, const void* C_in, int64_t ldc, const float* scale,
                     const int64_t* rows, const int64_t* cols, int64_t nsamples,
                     double* out, int64_t* acc_i64, int nthreads)
{
    if (K % 4 != 0 || check_types(dt_ab, dt_c)) return -1;
    for (int64_t s = 0; s < nsamples; ++s)
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dt_ab = dt_ab; j.dt_c = dt_c; j.M = M; j.N = N; j.K = K; j.ldb = ldb; j.ldc = ldc;
    j.alpha = alpha; j.beta = beta; j.values = values; j.meta = meta; j.B = B; j.C_in = C_in;
    j.scale = scale; j.out = out; j.acc_i64 = acc_i64;
    j.rows = rows; j.cols = cols; j.nsamples = nsamples;
    return parallel_for(&j, nsamples, nthreads, run_samples);
}

static int parallel_for(job_t* base, int64_t total, int nthreads, void* (*fn)(void*));
static int check_types(int dt_ab, int dt_c);

/* The transposed product (see above), all K x N outputs; out and acc_i64 are
 * N*K, (k, n) at [n*K + k].  Returns the threads used, or -1 on bad arguments. */
int orc_spmm_t(int dt_ab, int dt_c, int64_t M, int64_t N, int64_t K, double alpha,
               const void* values, const uint8_t* meta, const void* B, int64_t ldb,
               double beta, const void* C_in, int64_t ldc, double* out, int64_t* acc_i64, int nthreads)
{
    if (K % 4 != 0 || check_types(dt_ab, dt_c)) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dt_ab = dt_ab; j.dt_c = dt_c; j.M = M; j.N = N; j.K = K; j.ldb = ldb; j.ldc = ldc;
    j.alpha = alpha; j.beta = beta; j.values = values; j.meta = meta; j.B = B; j.C_in = C_in;
    j.out = out; j.acc_i64 = acc_i64;
    return parallel_for(&j, K, nthreads, run_rows_t);
}

/* Selected outputs (ks[s], ns[s]) of the transposed product; out[s]. */
int orc_spmm_t_sampled(int dt_ab, int dt_c, int64_t M, int64_t N, int64_t K, double alpha,
                       const void* values, const uint8_t* meta, const void* B, int64_t ldb,
                       double beta, const void* C_in, int64_t ldc, const int64_t* ks, const int64_t* ns,
                       int64_t nsamples, double* out, int64_t* acc_i64, int nthreads)
{
    if (K % 4 != 0 || check_types(dt_ab, dt_c)) return -1;
    for (int64_t s = 0; s < nsamples; ++s)
        if (ks[s] < 0 || ks[s] >= K || ns[s] < 0 || ns[s] >= N) return -1;
    job_t j;
    memset(&j, 0, sizeof j);
    j.dt_ab = dt_ab; j.dt_c = dt_c; j.M = M; j.N = N; j.K = K; j.ldb = ldb; j.ldc = ldc;
    j.alpha = alpha; j.beta = beta; j.values = values; j.meta = meta; j.B = B; j.C_in = C_in;
    j.out = out; j.acc_i64 = acc_i64;
    j.rows = ks; j.cols = ns; j.nsamples = nsamples;
    return parallel_for(&j, nsamples, nthreads, run_samples_t);
}

/* Threads a call with nthreads = 0 would use (for reporting). */
int orc_default_threads(void) { return thread_count(0); }
