/*
 * Oracle for the preshuffled-weight GEMM: a plain, slow, obviously correct
 * CPU implementation in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (aiter PR "FlyDSL split-K preshuffle decode GEMM for
 * small-M shapes (FP8 + MX, gfx950/gfx942)", Summary and What's included;
 * FlyDSL PR "Enable the gmem->LDS async copy for f16/bf16 preshuffle GEMM",
 * Summary):
 *
 *     y[m,n] = sum_{k=k0}^{k1-1} Ad[m,k] * Bd[n,k]        (fp64, k ascending)
 *
 * where Ad, Bd are the dequantised operands of the scale mode:
 *   BF16         Ad = A                               (bf16 bit pattern)
 *   FP8_TENSOR   Ad = e4m3(a); the per-tensor factor a_s*b_s is applied
 *                after the sum when `tensor_scale` is set (the split-K page
 *                downcasts and scales once, at the final store)
 *   FP8_BLOCK128 Ad = e4m3(a) * a_s[m][k/128],  Bd = e4m3(b) * b_s[n/128][k/128]
 *   MXFP8        Ad = e4m3(a) * 2^(a_sf[m][k/128]-127)     ("mx128")
 *   MXFP4        Ad = e2m1(a) * 2^(a_sf[m][k/32]-127), two e2m1 codes per
 *                byte, low nibble = even k
 *   MXFP8_B32    Ad = e4m3(a) * 2^(a_sf[m][k/32]-127)      (the OCP MX block of
 *                32 elements, next to the pages' 128-element "mx128")
 * and the same for B with n in place of m, except
 *   MXFP4_FP8A   Ad as MXFP8_B32, Bd as MXFP4: fp8 activations against fp4
 *                weights, both with one E8M0 per 32 K (the "MXFP4 fp8-A"
 *                preshuffle-GEMM test cases named in the FlyDSL PR "Enable
 *                the gmem->LDS async copy for f16/bf16 preshuffle GEMM",
 *                Testing)
 *
 * Encodings are decoded from their bit fields through 256-entry tables built
 * once (OCP 8-bit floating point E4M3 "fn", OCP FP4 E2M1, E8M0, bfloat16).
 *
 * Parity pins (the tests check this file against them, not against itself):
 * exhaustive table comparison with independent dtype libraries, exact
 * rational brute force on tiny shapes, identity and all-ones closed forms,
 * exactness of split sums, and the bijectivity of the layout spec below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    ORC_BF16 = 0,
    ORC_FP8_TENSOR = 1,
    ORC_FP8_BLOCK128 = 2,
    ORC_MXFP8 = 3,
    ORC_MXFP4 = 4,
    ORC_MXFP8_B32 = 5,
    ORC_MXFP4_FP8A = 6
};

/* ---------------------------------------------------------------- decoding */

/* OCP E4M3 "fn": s.eeee.mmm, bias 7, no infinities, s.1111.111 is NaN. */
static double decode_e4m3_bits(unsigned c)
{
    unsigned s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m, -9);                 /* m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8u + m), (int)e - 10); /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* OCP E2M1: s.ee.m, bias 1; values 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static double decode_e2m1_bits(unsigned nib)
{
    unsigned s = (nib >> 3) & 1u, e = (nib >> 1) & 3u, m = nib & 1u;
    double v;
    if (e == 0u)
        v = 0.5 * (double)m;                      /* m/2 * 2^(1-1) */
    else
        v = ldexp((double)(2u + m), (int)e - 2);  /* (1+m/2) * 2^(e-1) */
    return s ? -v : v;
}

/* E8M0: an unsigned biased exponent, 2^(c-127); 0xFF is NaN. */
static double decode_e8m0_bits(unsigned c)
{
    if (c == 255u)
        return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* bfloat16: s.eeeeeeee.mmmmmmm, bias 127. */
static double decode_bf16_bits(unsigned h)
{
    unsigned s = (h >> 15) & 1u, e = (h >> 7) & 255u, m = h & 127u;
    double v;
    if (e == 255u)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0u)
        v = ldexp((double)m, -133);                 /* m/128 * 2^-126 */
    else
        v = ldexp((double)(128u + m), (int)e - 134); /* (1+m/128) * 2^(e-127) */
    return s ? -v : v;
}

static double T_E4M3[256], T_E2M1[16], T_E8M0[256];
static pthread_once_t tables_once = PTHREAD_ONCE_INIT;

static void build_tables(void)
{
    for (unsigned c = 0; c < 256u; ++c) {
        T_E4M3[c] = decode_e4m3_bits(c);
        T_E8M0[c] = decode_e8m0_bits(c);
    }
    for (unsigned c = 0; c < 16u; ++c)
        T_E2M1[c] = decode_e2m1_bits(c);
}

static void ensure_tables(void) { pthread_once(&tables_once, build_tables); }

/* Table dumps, for the exhaustive comparison against other decoders. */
void orc_table_e4m3(double *out) { ensure_tables(); memcpy(out, T_E4M3, sizeof T_E4M3); }
void orc_table_e2m1(double *out) { ensure_tables(); memcpy(out, T_E2M1, sizeof T_E2M1); }
void orc_table_e8m0(double *out) { ensure_tables(); memcpy(out, T_E8M0, sizeof T_E8M0); }
void orc_decode_bf16(const uint16_t *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode_bf16_bits(in[i]);
}

/* ------------------------------------------------------ element accessors */

typedef struct {
    int mode;
    int64_t M, N, K;
    const void *A, *B, *a_scale, *b_scale;
    int64_t k0, k1;
    const int64_t *rows;
    int64_t n_rows;
    int tensor_scale;
    double *out;
    int64_t row_begin, row_end; /* range of `rows` indices for one thread */
} orc_job;

/* Number of scale columns per row: ceil(K / block); ceil so that tiny cases
 * with a partial block (K < block) index correctly. */
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* e4m3 code [rows][K] times 2^(scale-127), one E8M0 per 32 K. */
static double e4m3_e8m0_32(const void *X, const void *S, int64_t K, int64_t r, int64_t k)
{
    const int64_t kb = ceil_div(K, 32);
    const double s = T_E8M0[((const uint8_t *)S)[r * kb + k / 32]];
    return T_E4M3[((const uint8_t *)X)[r * K + k]] * s;
}

/* e2m1 codes packed two per byte [rows][K/2] (low nibble = even k) times
 * 2^(scale-127), one E8M0 per 32 K. */
static double e2m1_e8m0_32(const void *X, const void *S, int64_t K, int64_t r, int64_t k)
{
    const int64_t kb = ceil_div(K, 32);
    const double s = T_E8M0[((const uint8_t *)S)[r * kb + k / 32]];
    const uint8_t byte = ((const uint8_t *)X)[r * ceil_div(K, 2) + k / 2];
    const unsigned nib = (k & 1) ? (byte >> 4) : (byte & 15u);
    return T_E2M1[nib] * s;
}

/* Dequantised value of operand X (A or B) at (r, k).  `is_b` selects the
 * B-side block-scale indexing (128x128 blocks for FP8_BLOCK128). */
static double dequant(const orc_job *j, int is_b, int64_t r, int64_t k)
{
    const void *X = is_b ? j->B : j->A;
    const void *S = is_b ? j->b_scale : j->a_scale;
    const int64_t K = j->K;
    switch (j->mode) {
    case ORC_BF16:
        return decode_bf16_bits(((const uint16_t *)X)[r * K + k]);
    case ORC_FP8_TENSOR:
        return T_E4M3[((const uint8_t *)X)[r * K + k]];
    case ORC_FP8_BLOCK128: {
        const int64_t kb = ceil_div(K, 128);
        const int64_t sr = is_b ? r / 128 : r;
        const double s = (double)((const float *)S)[sr * kb + k / 128];
        return T_E4M3[((const uint8_t *)X)[r * K + k]] * s;
    }
    case ORC_MXFP8: {
        const int64_t kb = ceil_div(K, 128);
        const double s = T_E8M0[((const uint8_t *)S)[r * kb + k / 128]];
        return T_E4M3[((const uint8_t *)X)[r * K + k]] * s;
    }
    case ORC_MXFP8_B32:
        return e4m3_e8m0_32(X, S, K, r, k);
    case ORC_MXFP4:
        return e2m1_e8m0_32(X, S, K, r, k);
    case ORC_MXFP4_FP8A: /* fp8 activations, fp4 weights */
        return is_b ? e2m1_e8m0_32(X, S, K, r, k) : e4m3_e8m0_32(X, S, K, r, k);
    }
    return NAN;
}

static void *gemm_rows(void *arg)
{
    orc_job *j = (orc_job *)arg;
    const int64_t K = j->K;
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double ts = 1.0;
    if (j->mode == ORC_FP8_TENSOR && j->tensor_scale)
        ts = (double)*(const float *)j->a_scale * (double)*(const float *)j->b_scale;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        const int64_t m = j->rows ? j->rows[i] : i;
        for (int64_t k = j->k0; k < j->k1; ++k)
            arow[k] = dequant(j, 0, m, k);
        for (int64_t n = 0; n < j->N; ++n) {
            double acc = 0.0;
            for (int64_t k = j->k0; k < j->k1; ++k)
                acc += arow[k] * dequant(j, 1, n, k);
            j->out[i * j->N + n] = acc * ts;
        }
    }
    free(arow);
    return NULL;
}

/*
 * y[i][n] for the rows `rows[0..n_rows)` (all M rows, in order, when rows is
 * NULL), summed over k in [k0, k1).  Returns 0, or -1 on a bad argument.
 * Rows are shared out over `threads` POSIX threads; each output element is
 * one sequential fp64 sum in k order, so the result does not depend on the
 * thread count.
 */
int orc_gemm(int mode, int64_t M, int64_t N, int64_t K,
             const void *A, const void *B, const void *a_scale, const void *b_scale,
             int64_t k0, int64_t k1, const int64_t *rows, int64_t n_rows,
             int tensor_scale, double *out, int threads)
{
    ensure_tables();
    if (mode < ORC_BF16 || mode > ORC_MXFP4_FP8A || M < 0 || N < 0 || K < 0)
        return -1;
    if (k0 < 0 || k1 > K || k0 > k1)
        return -1;
    if ((mode == ORC_MXFP4 || mode == ORC_MXFP4_FP8A) && (K % 2) != 0)
        return -1;
    if (!rows)
        n_rows = M;
    for (int64_t i = 0; rows && i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= M)
            return -1;
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (n_rows < threads)
        threads = n_rows > 0 ? (int)n_rows : 1;

    orc_job base = {mode, M, N, K, A, B, a_scale, b_scale, k0, k1,
                    rows, n_rows, tensor_scale, out, 0, 0};
    orc_job jobs[256];
    pthread_t tid[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = base;
        jobs[t].row_begin = n_rows * t / threads;
        jobs[t].row_end = n_rows * (t + 1) / threads;
    }
    for (int t = 1; t < threads; ++t)
        pthread_create(&tid[t], NULL, gemm_rows, &jobs[t]);
    gemm_rows(&jobs[0]);
    for (int t = 1; t < threads; ++t)
        pthread_join(tid[t], NULL);
    return 0;
}

/* ---------------------------------------------------------- split ranges */

/*
 * K is cut into units of one 128-byte K-slab (64 bf16, 128 fp8 or 256 fp4
 * elements).  Split s of S gets floor(U/S) units, plus one more when
 * s < U mod S; ranges are contiguous and in split order.  The pages do not
 * say how the remainder is shared out; this is the reading used throughout.
 * Writes the element range [k_begin, k_end) of split s.
 */
int orc_splitk_range(int mode, int64_t K, int S, int s, int64_t *k_begin, int64_t *k_end)
{
    int64_t per_unit;
    if (mode == ORC_BF16)
        per_unit = 64;
    else if (mode == ORC_MXFP4)
        per_unit = 256;
    else if ((mode >= ORC_FP8_TENSOR && mode <= ORC_MXFP8) || mode == ORC_MXFP8_B32 || mode == ORC_MXFP4_FP8A)
        per_unit = 128; /* MXFP4_FP8A: one 128-byte slab of the fp8 A */
    else
        return -1;
    if (S < 1 || s < 0 || s >= S || K < 0 || K % per_unit != 0)
        return -1;
    const int64_t U = K / per_unit, q = U / S, r = U % S;
    const int64_t u0 = (int64_t)s * q + (s < r ? s : r);
    const int64_t u1 = u0 + q + (s < r ? 1 : 0);
    *k_begin = u0 * per_unit;
    *k_end = u1 * per_unit;
    return 0;
}

/* --------------------------------------------------- weight layout (spec) */

/*
 * The preshuffled weight image.  B is viewed as bytes, N rows of Kb bytes
 * (Kb = 2K for bf16, K for fp8, K/2 for packed fp4).  It is cut into slabs
 * of 128 rows x 128 bytes; slab (nb, kb) is stored at slab index
 * nb * (Kb/128) + kb, and inside a slab the 16-byte chunk c of row r goes to
 * byte offset r*128 + ((c XOR (r mod 8)) * 16).  The pages leave the layout
 * to the implementation; the only contract is that it is a bijection whose
 * inverse restores B exactly.
 */
int orc_preshuffle_b(const uint8_t *B, int64_t N, int64_t Kb, uint8_t *out)
{
    if (N % 128 != 0 || Kb % 128 != 0 || N < 0 || Kb < 0)
        return -1;
    const int64_t KB = Kb / 128;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t kbyte = 0; kbyte < Kb; kbyte += 16) {
            const int64_t nb = n / 128, r = n % 128, kb = kbyte / 128, c = (kbyte % 128) / 16;
            const int64_t dst = ((nb * KB + kb) * 128 + r) * 128 + ((c ^ (r % 8)) * 16);
            memcpy(out + dst, B + n * Kb + kbyte, 16);
        }
    return 0;
}

int orc_unshuffle_b(const uint8_t *in, int64_t N, int64_t Kb, uint8_t *B)
{
    if (N % 128 != 0 || Kb % 128 != 0 || N < 0 || Kb < 0)
        return -1;
    const int64_t KB = Kb / 128;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t kbyte = 0; kbyte < Kb; kbyte += 16) {
            const int64_t nb = n / 128, r = n % 128, kb = kbyte / 128, c = (kbyte % 128) / 16;
            const int64_t src = ((nb * KB + kb) * 128 + r) * 128 + ((c ^ (r % 8)) * 16);
            memcpy(B + n * Kb + kbyte, in + src, 16);
        }
    return 0;
}

/*
 * The MXFP4_FP8A weight image: B as packed fp4 bytes, N rows of Kb = K/2
 * bytes, cut into blocks of 128 rows x 64 bytes (128 K of fp4), block
 * (nb, u) at index nb * (Kb/64) + u, row r of the block at byte r*64, no
 * swizzle.
 */
int orc_block64_b(const uint8_t *B, int64_t N, int64_t Kb, uint8_t *out)
{
    if (N % 128 != 0 || Kb % 64 != 0 || N < 0 || Kb < 0)
        return -1;
    const int64_t U = Kb / 64;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t u = 0; u < U; ++u)
            memcpy(out + ((n / 128) * U + u) * 8192 + (n % 128) * 64, B + n * Kb + u * 64, 64);
    return 0;
}

int orc_unblock64_b(const uint8_t *in, int64_t N, int64_t Kb, uint8_t *B)
{
    if (N % 128 != 0 || Kb % 64 != 0 || N < 0 || Kb < 0)
        return -1;
    const int64_t U = Kb / 64;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t u = 0; u < U; ++u)
            memcpy(B + n * Kb + u * 64, in + ((n / 128) * U + u) * 8192 + (n % 128) * 64, 64);
    return 0;
}

/* --------------------------------------------------------- final rounding */

/* bf16 round-to-nearest-even of an fp32 value, from its bit pattern. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Round fp64 results to fp32 and then to bf16 (RNE both steps). */
void orc_round_bf16(const double *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)in[i]);
}

/* ------------------------------------------- MX scale image (layout spec) */

/*
 * The weight scale image of the MX modes: 512-byte atoms whose byte
 * 16*(r%32) + 4*(r/32) + j belongs to row nb*128 + r of 128-row tile nb.
 *   MXFP4, MXFP8_B32 (and the fp4 weights of MXFP4_FP8A, whose slab is 128 K
 *   like MXFP8_B32's): for each 128-byte K slab u and each atom a of the slab
 *   (two per slab for MXFP4, one otherwise), byte j is the scale of the 32-K
 *   block (u*atoms + a)*4 + j.  sf is [N][K/32].
 *   MXFP8 (one scale per 128 K): for each group g of four consecutive slabs,
 *   byte j is the scale of slab 4g + j (zero past the last slab).  sf is
 *   [N][K/128].  (The layout is the implementation's own; packing four
 *   slabs lets the kernels copy an atom into the tensor memory once per four
 *   slabs, the MMA picking byte j by its scale-factor id.)
 */
int orc_sf_image(int mode, const uint8_t *sf, int64_t N, int64_t K, uint8_t *out)
{
    if (mode == ORC_MXFP4_FP8A)
        mode = ORC_MXFP8_B32;
    if ((mode != ORC_MXFP8 && mode != ORC_MXFP4 && mode != ORC_MXFP8_B32) || N % 128 != 0)
        return -1;
    if (mode == ORC_MXFP8) {
        if (K % 128 != 0)
            return -1;
        const int64_t KB = K / 128, G = (KB + 3) / 4;
        memset(out, 0, (size_t)((N / 128) * G * 512));
        for (int64_t n = 0; n < N; ++n)
            for (int64_t u = 0; u < KB; ++u) {
                const int64_t nb = n / 128, r = n % 128;
                out[(nb * G + u / 4) * 512 + 16 * (r % 32) + 4 * (r / 32) + u % 4] = sf[n * KB + u];
            }
        return 0;
    }
    const int64_t slab_k = mode == ORC_MXFP4 ? 256 : 128;
    if (K % slab_k != 0)
        return -1;
    const int64_t atoms = mode == ORC_MXFP4 ? 2 : 1;
    const int64_t slabs = K / slab_k;
    const int64_t cols = K / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < K / 32; ++q) {          /* 32-K block index */
            const int64_t nb = n / 128, r = n % 128;
            const int64_t u = q / (4 * atoms), a = (q / 4) % atoms, j = q % 4;
            const int64_t atom = (nb * slabs + u) * atoms + a;
            out[atom * 512 + 16 * (r % 32) + 4 * (r / 32) + j] = sf[n * cols + q];
        }
    return 0;
}
