/*
 * CPU oracle for the W4A16 group-quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (plain definitions, fp64 throughout, written for reading,
 * not for speed):
 *
 *   w[n,k] = (q[n,k] - z[n,j]) * s[n,j],   j = floor(k / g)
 *   y[m,n] = sum_k x[m,k] * w[n,k]
 *
 * Sources:
 *  - 4-bit weights with fp16 activations: Marlin post ("FP16xINT4 kernel"),
 *    and lmdeploy PR #202 "Blazing fast W4A16 inference".
 *  - Group-wise quantization along K with a group size: lmdeploy PR #202
 *    (converter flags --model_format awq --group_size 128) and torchchat
 *    issue #1362 ('linear:int4': {'groupsize': 256}).
 *  - A last group narrower than g, handled rather than padded or skipped:
 *    torchchat issue #1362, option 2 ("groupwise GEMM with a last group
 *    that's not a full group"), motivated there by a 288x288 weight with
 *    group size 256.
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of the repository):
 *  - the range of each group includes zero: lo = min(0, min w), hi = max(0, max w);
 *  - s is r/15 rounded to fp16 (round-to-nearest-even straight from fp64),
 *    then raised by one fp16 step if 15*s < r, so 15*s >= r always;
 *  - a group with r == 0 gets s = 1, z = 0 and all codes 0;
 *  - all rounding to integers is round-half-to-even;
 *  - codes are packed 8 per uint32 along K, code k = 8c + i in bits
 *    4i..4i+3 of word c; zeros are packed the same way along groups;
 *    padding nibbles are 0;
 *  - non-finite weights are rejected;
 *  - bf16 weights, scales and activations (the 'bf16' precision torchchat
 *    issue #1362 runs int4 quantization with) follow the same steps, with
 *    every value of that type widened exactly and s rounded to bfloat16;
 *  - the symmetric form fixes z at 8 and takes the range [-max|w|, max|w|]
 *    (r = 2 max|w|); a group of zeros gets s = 1, z = 8, q = 8.
 *
 * Compile with -ffp-contract=off (no fused multiply-add) and no fast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16, from the format's definition: 1 sign bit, 5      */
/* exponent bits (bias 15), 10 fraction bits.                          */
/* ------------------------------------------------------------------ */

double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a non-negative integral-plus-fraction double to an integer, ties to even. */
static double round_half_even(double v)
{
    double fl = floor(v);
    double d = v - fl; /* exact: v and fl share the binade or fl == 0 */
    if (d > 0.5)
        return fl + 1.0;
    if (d < 0.5)
        return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Signed round-half-even to an integer value (for quotients of either sign). */
static double rne_int(double v)
{
    return v < 0 ? -round_half_even(-v) : round_half_even(v);
}

/* fp64 -> binary16, round to nearest, ties to even, in one step. */
uint16_t orc_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (a >= 65520.0) /* 65504 + half a step rounds (to even) up to 2^16: overflow */
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1; /* a in [2^e, 2^(e+1)) */
    if (e < -14) {
        /* subnormal range: multiples of 2^-24 */
        double n = round_half_even(ldexp(a, 24));
        return sign | (uint16_t)n; /* n == 1024 is the smallest normal, encoded alike */
    }
    double n = round_half_even(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (n == 2048.0) {
        n = 1024.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7c00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* ------------------------------------------------------------------ */
/* bfloat16, from the format's definition: 1 sign bit, 8 exponent bits */
/* (bias 127), 7 fraction bits.                                        */
/* ------------------------------------------------------------------ */

double orc_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* subnormal: f * 2^-133 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* fp64 -> bfloat16, round to nearest, ties to even, in one step. */
uint16_t orc_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7fc0;
    /* halfway between the largest finite value (2 - 2^-7) * 2^127 and 2^128 rounds (to even) up */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127))
        return sign | 0x7f80;
    if (a == 0.0)
        return sign;
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1; /* a in [2^e, 2^(e+1)) */
    if (e < -126) {
        /* subnormal range: multiples of 2^-133 */
        double n = round_half_even(ldexp(a, 133));
        return sign | (uint16_t)n; /* n == 128 is the smallest normal, encoded alike */
    }
    double n = round_half_even(ldexp(a, 7 - e)); /* in [128, 256] */
    if (n == 256.0) {
        n = 128.0;
        e += 1;
    }
    if (e > 127)
        return sign | 0x7f80;
    return sign | (uint16_t)(((e + 127) << 7) | ((int)n - 128));
}

/* The 16-bit value types of weights, scales and activations: 0 = fp16, 1 = bf16. */
static double dt_to_double(uint16_t bits, int dtype)
{
    return dtype ? orc_bf16_to_double(bits) : orc_half_to_double(bits);
}

static uint16_t dt_from_double(double v, int dtype)
{
    return dtype ? orc_double_to_bf16(v) : orc_double_to_half(v);
}

static uint16_t dt_one(int dtype) { return dtype ? 0x3f80 : 0x3c00; }

/* ------------------------------------------------------------------ */
/* Quantization (encoding step).                                       */
/* ------------------------------------------------------------------ */

/* The least positive value of the type that is >= r / 15: round r / 15 to nearest (ties to even)
 * straight from fp64, then one step up if 15 times that is still below r. */
static uint16_t scale_at_least(double r, int dtype)
{
    uint16_t sb = dt_from_double(r / 15.0, dtype);
    if (dt_to_double(sb, dtype) * 15.0 < r) /* exact product: at most 11 + 4 significant bits */
        sb = (uint16_t)(sb + 1);            /* next value up (sb is positive, finite) */
    return sb;
}

/*
 * W [N,K] bits of type `dtype` -> codes q [N,K] (0..15), scales s [N,G] (bits of `dtype`),
 * zeros z [N,G] (0..15). symmetric == 0: the range of each group includes zero,
 * [min(0, min w), max(0, max w)], and z places zero on the code grid; symmetric == 1: the
 * range is [-max|w|, max|w|] and z is 8 for every group.
 * Returns 0, or -1 for bad arguments, -2 for a non-finite weight.
 */
int orc_quantize_ex(const uint16_t *W, int64_t N, int64_t K, int32_t g, int32_t dtype, int32_t symmetric,
                    uint8_t *q, uint16_t *s, uint8_t *z)
{
    if (N < 1 || K < 1 || g < 1 || dtype < 0 || dtype > 1 || symmetric < 0 || symmetric > 1)
        return -1;
    int64_t G = (K + g - 1) / g;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t j = 0; j < G; ++j) {
            int64_t k0 = j * g;
            int64_t k1 = k0 + g < K ? k0 + g : K; /* last group may be narrower */
            double lo = 0.0, hi = 0.0;
            for (int64_t k = k0; k < k1; ++k) {
                double w = dt_to_double(W[n * K + k], dtype);
                if (!isfinite(w))
                    return -2;
                if (w < lo)
                    lo = w;
                if (w > hi)
                    hi = w;
            }
            if (symmetric) {
                double amax = hi > -lo ? hi : -lo;
                lo = -amax;
                hi = amax;
            }
            double r = hi - lo;
            uint16_t sb;
            int zj;
            if (r == 0.0) {
                sb = dt_one(dtype);
                zj = symmetric ? 8 : 0;
            } else {
                sb = scale_at_least(r, dtype);
                if (symmetric) {
                    zj = 8;
                } else {
                    double zz = rne_int(-lo / dt_to_double(sb, dtype));
                    zj = zz < 0 ? 0 : (zz > 15 ? 15 : (int)zz);
                }
            }
            s[n * G + j] = sb;
            z[n * G + j] = (uint8_t)zj;
            double sv = dt_to_double(sb, dtype);
            for (int64_t k = k0; k < k1; ++k) {
                int qk = zj; /* r == 0: every weight is 0 and encodes as z */
                if (r != 0.0) {
                    double w = dt_to_double(W[n * K + k], dtype);
                    double t = rne_int(w / sv) + (double)zj;
                    qk = t < 0 ? 0 : (t > 15 ? 15 : (int)t);
                }
                q[n * K + k] = (uint8_t)qk;
            }
        }
    }
    return 0;
}

/* fp16 weights, range including zero (the default form). */
int orc_quantize(const uint16_t *W, int64_t N, int64_t K, int32_t g, uint8_t *q, uint16_t *s, uint8_t *z)
{
    return orc_quantize_ex(W, N, K, g, 0, 0, q, s, z);
}

/* ------------------------------------------------------------------ */
/* Canonical packing: 8 nibbles per uint32, element i at bits 4i..4i+3 */
/* ------------------------------------------------------------------ */

/* v [rows, cols] bytes (0..15) -> out [rows, ceil(cols/8)] uint32. */
void orc_pack_nibbles(const uint8_t *v, int64_t rows, int64_t cols, uint32_t *out)
{
    int64_t cw = (cols + 7) / 8;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cw; ++c) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i) {
                int64_t e = 8 * c + i;
                uint32_t nib = e < cols ? (uint32_t)(v[r * cols + e] & 0xf) : 0u;
                word |= nib << (4 * i);
            }
            out[r * cw + c] = word;
        }
}

void orc_unpack_nibbles(const uint32_t *in, int64_t rows, int64_t cols, uint8_t *v)
{
    int64_t cw = (cols + 7) / 8;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t e = 0; e < cols; ++e)
            v[r * cols + e] = (uint8_t)((in[r * cw + e / 8] >> (4 * (e % 8))) & 0xf);
}

/* ------------------------------------------------------------------ */
/* Tile layout ("repacked" weights), restated from its specification:  */
/*                                                                     */
/*  TN = 128 rows per n-tile, TK = 64 codes per k-block.               */
/*  NT = ceil(N/128), KB = ceil(K/64), G = ceil(K/g).                  */
/*  Code region, NT*KB tiles of 4096 bytes, tile (t,b) at byte         */
/*  (t*KB + b)*4096. In a tile, the little-endian uint32 at byte       */
/*  h*2048 + r*16 + 4*i  (h<2, r<128, i<4) holds the 8 codes of row    */
/*  n = 128t + r at k = 64b + 32h + 8i + e (e<8); code e sits at       */
/*  nibble 4*(e%2) + e/2. Codes at n >= N or k >= K are 0.             */
/*  Group region after it, NT*G records of 320 bytes, record (t,j) at  */
/*  NT*KB*4096 + (t*G + j)*320: bytes 2r..2r+1 hold the fp16 scale of  */
/*  row 128t + r and group j; byte 256 + r/2 holds its zero in the     */
/*  low nibble (r even) or high nibble (r odd). Rows >= N hold zeros.  */
/* ------------------------------------------------------------------ */

#define ORC_TN 128
#define ORC_TK 64
#define ORC_TILE_BYTES 4096
#define ORC_REC_BYTES 320

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t orc_repacked_bytes(int64_t N, int64_t K, int32_t g)
{
    int64_t NT = cdiv(N, ORC_TN), KB = cdiv(K, ORC_TK), G = cdiv(K, g);
    return NT * KB * ORC_TILE_BYTES + NT * G * ORC_REC_BYTES;
}

static int nib_pos(int e) { return 4 * (e % 2) + e / 2; }

/* canonical (qw [N,ceil(K/8)], scales [N,G] fp16 bits, zw [N,ceil(G/8)]) -> out */
void orc_repack(const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                int64_t N, int64_t K, int32_t g, uint8_t *out)
{
    int64_t NT = cdiv(N, ORC_TN), KB = cdiv(K, ORC_TK), G = cdiv(K, g);
    int64_t Kw = cdiv(K, 8), Gw = cdiv(G, 8);
    memset(out, 0, (size_t)orc_repacked_bytes(N, K, g));
    for (int64_t t = 0; t < NT; ++t)
        for (int64_t b = 0; b < KB; ++b)
            for (int h = 0; h < 2; ++h)
                for (int r = 0; r < ORC_TN; ++r)
                    for (int i = 0; i < 4; ++i) {
                        int64_t n = ORC_TN * t + r;
                        uint32_t word = 0;
                        for (int e = 0; e < 8; ++e) {
                            int64_t k = ORC_TK * b + 32 * h + 8 * i + e;
                            uint32_t code = 0;
                            if (n < N && k < K)
                                code = (qw[n * Kw + k / 8] >> (4 * (k % 8))) & 0xf;
                            word |= code << (4 * nib_pos(e));
                        }
                        uint8_t *p = out + (t * KB + b) * ORC_TILE_BYTES + h * 2048 + r * 16 + 4 * i;
                        p[0] = (uint8_t)(word & 0xff);
                        p[1] = (uint8_t)((word >> 8) & 0xff);
                        p[2] = (uint8_t)((word >> 16) & 0xff);
                        p[3] = (uint8_t)((word >> 24) & 0xff);
                    }
    uint8_t *meta = out + NT * KB * ORC_TILE_BYTES;
    for (int64_t t = 0; t < NT; ++t)
        for (int64_t j = 0; j < G; ++j) {
            uint8_t *rec = meta + (t * G + j) * ORC_REC_BYTES;
            for (int r = 0; r < ORC_TN; ++r) {
                int64_t n = ORC_TN * t + r;
                if (n >= N)
                    continue;
                uint16_t sb = scales[n * G + j];
                rec[2 * r] = (uint8_t)(sb & 0xff);
                rec[2 * r + 1] = (uint8_t)(sb >> 8);
                uint32_t zj = (zw[n * Gw + j / 8] >> (4 * (j % 8))) & 0xf;
                rec[256 + r / 2] |= (uint8_t)(zj << (4 * (r % 2)));
            }
        }
}

/* Inverse of orc_repack, written as the reverse map (tile layout -> canonical). */
void orc_unrepack(const uint8_t *in, int64_t N, int64_t K, int32_t g,
                  uint32_t *qw, uint16_t *scales, uint32_t *zw)
{
    int64_t KB = cdiv(K, ORC_TK), G = cdiv(K, g);
    int64_t NT = cdiv(N, ORC_TN);
    int64_t Kw = cdiv(K, 8), Gw = cdiv(G, 8);
    memset(qw, 0, sizeof(uint32_t) * (size_t)(N * Kw));
    memset(zw, 0, sizeof(uint32_t) * (size_t)(N * Gw));
    for (int64_t n = 0; n < N; ++n) {
        int64_t t = n / ORC_TN;
        int r = (int)(n % ORC_TN);
        for (int64_t k = 0; k < K; ++k) {
            int64_t b = k / ORC_TK;
            int within = (int)(k % ORC_TK);
            int h = within / 32, i = (within % 32) / 8, e = within % 8;
            const uint8_t *p = in + (t * KB + b) * ORC_TILE_BYTES + h * 2048 + r * 16 + 4 * i;
            uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                            ((uint32_t)p[3] << 24);
            uint32_t code = (word >> (4 * nib_pos(e))) & 0xf;
            qw[n * Kw + k / 8] |= code << (4 * (k % 8));
        }
        const uint8_t *meta = in + NT * KB * ORC_TILE_BYTES;
        for (int64_t j = 0; j < G; ++j) {
            const uint8_t *rec = meta + (t * G + j) * ORC_REC_BYTES;
            scales[n * G + j] = (uint16_t)(rec[2 * r] | (rec[2 * r + 1] << 8));
            uint32_t zj = (rec[256 + r / 2] >> (4 * (r % 2))) & 0xf;
            zw[n * Gw + j / 8] |= zj << (4 * (j % 8));
        }
    }
}

/* ------------------------------------------------------------------ */
/* Dequantize and multiply.                                            */
/* ------------------------------------------------------------------ */

/* One row of weights: w[k] = (q - z) * s, exact in fp64 (s of type `dtype`). */
static void dequant_row(const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                        int64_t n, int64_t K, int32_t g, int dtype, double *w)
{
    int64_t G = cdiv(K, g), Kw = cdiv(K, 8), Gw = cdiv(G, 8);
    for (int64_t k = 0; k < K; ++k) {
        int64_t j = k / g;
        int qk = (int)((qw[n * Kw + k / 8] >> (4 * (k % 8))) & 0xf);
        int zj = (int)((zw[n * Gw + j / 8] >> (4 * (j % 8))) & 0xf);
        double s = dt_to_double(scales[n * G + j], dtype);
        w[k] = (double)(qk - zj) * s;
    }
}

void orc_dequant_ex(const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                    int64_t N, int64_t K, int32_t g, int32_t dtype, double *w)
{
    for (int64_t n = 0; n < N; ++n)
        dequant_row(qw, scales, zw, n, K, g, dtype, w + n * K);
}

void orc_dequant(const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                 int64_t N, int64_t K, int32_t g, double *w)
{
    orc_dequant_ex(qw, scales, zw, N, K, g, 0, w);
}

struct gemm_job {
    const double *x; /* [R, K] fp64 rows of activations */
    int64_t R;
    const uint32_t *qw;
    const uint16_t *scales;
    const uint32_t *zw;
    int64_t N, K;
    int32_t g;
    int dtype;
    double *y; /* [R, N] */
    int64_t n_begin, n_end;
};

static void *gemm_worker(void *arg)
{
    struct gemm_job *jb = (struct gemm_job *)arg;
    double *w = (double *)malloc(sizeof(double) * (size_t)jb->K);
    if (!w)
        return (void *)1;
    for (int64_t n = jb->n_begin; n < jb->n_end; ++n) {
        dequant_row(jb->qw, jb->scales, jb->zw, n, jb->K, jb->g, jb->dtype, w);
        for (int64_t m = 0; m < jb->R; ++m) {
            const double *xm = jb->x + m * jb->K;
            double acc = 0.0;
            for (int64_t k = 0; k < jb->K; ++k)
                acc += xm[k] * w[k];
            jb->y[m * jb->N + n] = acc;
        }
    }
    free(w);
    return NULL;
}

/*
 * y[r, n] = sum_k x[rows[r], k] * w[n, k] for the listed activation rows
 * (rows == NULL: all M rows in order, R == M). x is [M, K] bits of type `dtype`
 * (0 fp16, 1 bf16; the scales are of the same type); y is fp64 [R, N], never
 * rounded. Threads split the n range. Returns 0, or -1 on allocation failure.
 */
int orc_gemm_rows_ex(const uint16_t *x, int64_t M, const int64_t *rows, int64_t R,
                     const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                     int64_t N, int64_t K, int32_t g, int32_t dtype, double *y, int nthreads)
{
    (void)M;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(R * K));
    if (!xd)
        return -1;
    for (int64_t r = 0; r < R; ++r) {
        int64_t src = rows ? rows[r] : r;
        for (int64_t k = 0; k < K; ++k)
            xd[r * K + k] = dt_to_double(x[src * K + k], dtype);
    }
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > N)
        nthreads = (int)N;
    struct gemm_job *jobs = (struct gemm_job *)calloc((size_t)nthreads, sizeof(struct gemm_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int rc = 0;
    if (!jobs || !th) {
        free(xd);
        free(jobs);
        free(th);
        return -1;
    }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (struct gemm_job){xd, R, qw, scales, zw, N, K, g, dtype, y,
                                    N * i / nthreads, N * (i + 1) / nthreads};
        if (pthread_create(&th[i], NULL, gemm_worker, &jobs[i]) != 0) {
            gemm_worker(&jobs[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < nthreads; ++i) {
        void *ret = NULL;
        if (th[i])
            pthread_join(th[i], &ret);
        if (ret)
            rc = -1;
    }
    free(xd);
    free(jobs);
    free(th);
    return rc;
}

/* fp16 activations and scales (the default form). */
int orc_gemm_rows(const uint16_t *x, int64_t M, const int64_t *rows, int64_t R,
                  const uint32_t *qw, const uint16_t *scales, const uint32_t *zw,
                  int64_t N, int64_t K, int32_t g, double *y, int nthreads)
{
    return orc_gemm_rows_ex(x, M, rows, R, qw, scales, zw, N, K, g, 0, y, nthreads);
}
