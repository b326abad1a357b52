/*
 * q1_oracle.c -- plain, slow, single-thread CPU oracle for the Q1_0 x q8_0
 * row dot product of 1-bit LLM decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, calls or reads this
 * file.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may use it.  It shares no code, header, table or constant with the CUDA
 * path: it defines the result the CUDA path must reproduce bit for bit.
 *
 * Source of the definition (bankML "docs/modules/gpu.md", section
 * "kernels.rs -- the Q1_0 kernels", first bullet; and "Advantages and
 * efficiency", bullet "Exact FMA only where needed"):
 *   - per 128-weight block, four 32-element sub-blocks;
 *   - eight lanes of exact integer sums, the i8 negation wrapping -128 to -128;
 *   - ab = d1*s on the first sub-block, ab = fma(d1, s, ab) after;
 *   - acc = fma(d0, ab, acc) with a single rounding;
 *   - the horizontal sum (a0+a4 + a2+a6) + (a1+a5 + a3+a7).
 * Each lane's chain over the blocks is independent (same section, second
 * bullet).  Scales are fp16, widened to f32 exactly (third/fourth bullets).
 *
 * Readings of what the pages leave open (each one is a stated contract):
 *   OPEN-1  block = 2-byte little-endian fp16 scale d0, then 16 bytes of sign
 *           bits; element j has bit (qs[j>>3] >> (j&7)) & 1; bit 1 = +d0,
 *           bit 0 = -d0.
 *   OPEN-2  q8_0 activation: per 32 values amax = max|x|, d = amax/127 (f32),
 *           id = d ? 1/d : 0 (f32), q = roundf(x*id) (half away from zero),
 *           stored scale = fp16 round-to-nearest-even of d.
 *   OPEN-4  lane accumulators start at +0.
 *   OPEN-5  lane l of a sub-block = its elements 4l..4l+3 (one i32 word of
 *           four i8 activation quants, "kernels.rs" bindings bullet).
 *   OPEN-6  horizontal sum read as ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)).
 *   OPEN-7  no flush-to-zero anywhere.
 *
 * The Q2_0 (ternary) section below carries its own readings, OPEN-10/11.
 *
 * Build: plain C11, -O2 -ffp-contract=off -fno-fast-math (no contraction of
 * a*b+c into an fma; every fma below is an explicit call to fmaf).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define Q1O_BLOCK 128      /* weights per Q1_0 block                        */
#define Q1O_BLOCK_BYTES 18 /* 2-byte fp16 scale + 16 bytes of sign bits     */
#define Q1O_QBLOCK 32      /* activation values per q8_0 scale (sub-block)   */
#define Q1O_LANES 8        /* accumulation lanes                             */
#define Q1O_CHUNK_ROWS 16  /* rows per claim in the threaded oracle          */

/* ------------------------------------------------------------------------ */
/* fp16 <-> f32                                                             */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bits -> f32, exact ("scales f16->f32, exact", kernels.rs
 * bullet on pack_q1_0).  Written from the binary16 definition:
 * value = (-1)^s * 2^(e-15) * (1 + m/1024) for 0 < e < 31,
 *         (-1)^s * 2^-14 * (m/1024)       for e == 0. */
float q1o_f16_to_f32(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0x1f)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexpf((float)m, -24);             /* subnormal: m * 2^-24 */
    else
        v = ldexpf((float)(m | 0x400), e - 25); /* (1024+m) * 2^(e-25) */
    return s ? -v : v;
}

/* f32 -> IEEE binary16 bits, round to nearest, ties to even, computed in
 * the integer domain (the approach vkML's "arch-shaders" page describes for
 * its f32->f16 narrowing).  Overflow gives +-Inf, NaN gives a quiet NaN. */
uint16_t q1o_f32_to_f16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    int e32 = (int)((u >> 23) & 0xff);
    uint32_t m32 = u & 0x7fffffu;

    if (e32 == 0xff)                       /* Inf or NaN */
        return sign | (m32 ? 0x7e00u : 0x7c00u);
    if (e32 == 0)                          /* f32 zero or subnormal: < 2^-126 */
        return sign;                       /* far below half an f16 ulp       */

    int E = e32 - 127;                     /* unbiased exponent               */
    uint32_t sig = m32 | 0x800000u;        /* 24-bit significand, value = sig*2^(E-23) */
    uint32_t mag;
    if (E >= -14) {
        /* normal f16 range (or overflow): keep 10 fraction bits */
        uint32_t keep = m32 >> 13;
        uint32_t rem = m32 & 0x1fffu;
        mag = ((uint32_t)(E + 15) << 10) + keep;
        if (rem > 0x1000u || (rem == 0x1000u && (keep & 1u)))
            mag += 1;                      /* carry may step into the exponent */
        if (E > 15 || mag >= 0x7c00u)
            mag = 0x7c00u;                 /* overflow to infinity            */
    } else {
        /* subnormal f16: units of 2^-24, value/2^-24 = sig * 2^(E+1) */
        int shift = -(E + 1);              /* >= 14 */
        if (shift > 24) {
            mag = 0;                       /* below 2^-25 before rounding: rounds to 0 */
        } else {
            uint32_t keep = sig >> shift;
            uint32_t rem = sig & ((1u << shift) - 1u);
            uint32_t half = 1u << (shift - 1);
            mag = keep;
            if (rem > half || (rem == half && (keep & 1u)))
                mag += 1;                  /* may become 0x400, the smallest normal */
        }
    }
    return sign | (uint16_t)mag;
}

/* Array forms of the two conversions (tests sweep many values at once). */
void q1o_f32_to_f16_rne_n(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = q1o_f32_to_f16_rne(x[i]);
}

void q1o_f16_to_f32_n(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = q1o_f16_to_f32(h[i]);
}

/* ------------------------------------------------------------------------ */
/* q8_0 activation quantization (OPEN-2)                                     */
/* ------------------------------------------------------------------------ */

/* x: n floats, n % 32 == 0.  q: n int8.  d: n/32 fp16 bits.
 * "pack_act repacks the q8_0 activation" (kernels.rs); the activation is
 * q8_0, i.e. one scale per 32 values, amax/127. */
void q1o_q8_quantize(const float *x, int64_t n, int8_t *q, uint16_t *d)
{
    for (int64_t b = 0; b < n / Q1O_QBLOCK; ++b) {
        const float *xb = x + b * Q1O_QBLOCK;
        float amax = 0.0f;
        for (int j = 0; j < Q1O_QBLOCK; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax)
                amax = a;
        }
        float dd = amax / 127.0f;
        float id = (dd != 0.0f) ? 1.0f / dd : 0.0f;
        d[b] = q1o_f32_to_f16_rne(dd);
        for (int j = 0; j < Q1O_QBLOCK; ++j) {
            float t = xb[j] * id;
            q[b * Q1O_QBLOCK + j] = (int8_t)(int)roundf(t);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q1_0 weight format (OPEN-1)                                               */
/* ------------------------------------------------------------------------ */

/* Sign bit of element j (0..127) of one 18-byte block. */
static int q1o_bit(const uint8_t *blk, int j)
{
    return (blk[2 + (j >> 3)] >> (j & 7)) & 1;
}

static uint16_t q1o_block_scale_bits(const uint8_t *blk)
{
    return (uint16_t)(blk[0] | (blk[1] << 8));
}

/* Dequantized weight (row r, column j) of a rows x n matrix stored as
 * rows*(n/128) consecutive 18-byte blocks, row-major: +d0 or -d0. */
float q1o_weight(const uint8_t *blocks, int64_t n, int64_t r, int64_t j)
{
    const uint8_t *blk = blocks + (r * (n / Q1O_BLOCK) + j / Q1O_BLOCK) * Q1O_BLOCK_BYTES;
    float d0 = q1o_f16_to_f32(q1o_block_scale_bits(blk));
    return q1o_bit(blk, (int)(j % Q1O_BLOCK)) ? d0 : -d0;
}

/* ------------------------------------------------------------------------ */
/* The row dot product                                                       */
/* ------------------------------------------------------------------------ */

/* i8 negation with the wrap the pages state: -(-128) stays -128. */
static int q1o_neg_i8(int v)
{
    int r = -v;
    return (r == 128) ? -128 : r;
}

/* Exact integer lane sum: sub-block k, lane l, of block blk, against the
 * activation quants qb of that block (128 values).  OPEN-5: lane l covers
 * elements 4l..4l+3 of the sub-block. */
static int32_t q1o_lane_sum(const uint8_t *blk, const int8_t *qb, int k, int l)
{
    int32_t s = 0;
    for (int i = 0; i < 4; ++i) {
        int j = Q1O_QBLOCK * k + 4 * l + i;
        int v = qb[j];
        s += q1o_bit(blk, j) ? v : q1o_neg_i8(v);
    }
    return s;
}

/* Variants exist ONLY for the negative-control test, which shows that the
 * parity checks are sensitive to the order of operations (bankML gpu.md,
 * "How it is verified": with a different rounding the check refuses the
 * card).  variant 0 is the contract; the others are deliberate departures:
 *   1: lane l takes elements {l, l+8, l+16, l+24} (strided lanes)
 *   2: horizontal sum strictly left to right over (a0,a4,a2,a6,a1,a5,a3,a7)
 *   3: outer step as a rounded multiply then a rounded add (no fma)
 *   4: lanes 0 and 1 exchanged in the horizontal sum pairing
 *      ((a1+a4)+(a2+a6)) + ((a0+a5)+(a3+a7)) */
static float q1o_dot_row_impl(const uint8_t *row_blocks, int64_t nb,
                              const int8_t *q, const uint16_t *d, int variant)
{
    float acc[Q1O_LANES];
    for (int l = 0; l < Q1O_LANES; ++l)
        acc[l] = 0.0f;                                   /* OPEN-4 */

    for (int64_t b = 0; b < nb; ++b) {                   /* blocks in order */
        const uint8_t *blk = row_blocks + b * Q1O_BLOCK_BYTES;
        const int8_t *qb = q + b * Q1O_BLOCK;
        float d0 = q1o_f16_to_f32(q1o_block_scale_bits(blk));
        for (int l = 0; l < Q1O_LANES; ++l) {
            float ab = 0.0f;
            for (int k = 0; k < 4; ++k) {
                int32_t s;
                if (variant == 1) {
                    s = 0;
                    for (int i = 0; i < 4; ++i) {
                        int j = Q1O_QBLOCK * k + l + 8 * i;
                        int v = qb[j];
                        s += q1o_bit(blk, j) ? v : q1o_neg_i8(v);
                    }
                } else {
                    s = q1o_lane_sum(blk, qb, k, l);
                }
                float d1 = q1o_f16_to_f32(d[b * 4 + k]);
                float t = (float)s;                       /* exact: |s| <= 512 */
                if (k == 0)
                    ab = d1 * t;                          /* exact in f32 */
                else
                    ab = fmaf(d1, t, ab);                 /* one rounding */
            }
            if (variant == 3) {
                float pr = d0 * ab;
                acc[l] = acc[l] + pr;
            } else {
                acc[l] = fmaf(d0, ab, acc[l]);            /* one rounding */
            }
        }
    }
    if (variant == 2)
        return ((((((acc[0] + acc[4]) + acc[2]) + acc[6]) + acc[1]) + acc[5]) + acc[3]) + acc[7];
    if (variant == 4)
        return ((acc[1] + acc[4]) + (acc[2] + acc[6])) + ((acc[0] + acc[5]) + (acc[3] + acc[7]));
    return ((acc[0] + acc[4]) + (acc[2] + acc[6])) + ((acc[1] + acc[5]) + (acc[3] + acc[7]));
}

/* One output row: row_blocks = nb 18-byte blocks, q = nb*128 int8,
 * d = nb*4 fp16 bits. */
float q1o_dot_row(const uint8_t *row_blocks, int64_t nb, const int8_t *q, const uint16_t *d)
{
    return q1o_dot_row_impl(row_blocks, nb, q, d, 0);
}

float q1o_dot_row_variant(const uint8_t *row_blocks, int64_t nb, const int8_t *q,
                          const uint16_t *d, int variant)
{
    return q1o_dot_row_impl(row_blocks, nb, q, d, variant);
}

/* The 8 lane accumulators of one row, before the horizontal sum (used by the
 * tests to check the error bound lane by lane). */
void q1o_dot_row_lanes(const uint8_t *row_blocks, int64_t nb, const int8_t *q,
                       const uint16_t *d, float *acc_out)
{
    float acc[Q1O_LANES] = {0};
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row_blocks + b * Q1O_BLOCK_BYTES;
        float d0 = q1o_f16_to_f32(q1o_block_scale_bits(blk));
        for (int l = 0; l < Q1O_LANES; ++l) {
            float ab = 0.0f;
            for (int k = 0; k < 4; ++k) {
                float d1 = q1o_f16_to_f32(d[b * 4 + k]);
                float t = (float)q1o_lane_sum(blk, q + b * Q1O_BLOCK, k, l);
                ab = (k == 0) ? d1 * t : fmaf(d1, t, ab);
            }
            acc[l] = fmaf(d0, ab, acc[l]);
        }
    }
    for (int l = 0; l < Q1O_LANES; ++l)
        acc_out[l] = acc[l];
}

/* Exact integer lane sums s[b][k][l] of one row (tests use them to build the
 * exact rational value of the dot product). */
void q1o_lane_sums(const uint8_t *row_blocks, int64_t nb, const int8_t *q, int32_t *s_out)
{
    for (int64_t b = 0; b < nb; ++b)
        for (int k = 0; k < 4; ++k)
            for (int l = 0; l < Q1O_LANES; ++l)
                s_out[(b * 4 + k) * Q1O_LANES + l] =
                    q1o_lane_sum(row_blocks + b * Q1O_BLOCK_BYTES, q + b * Q1O_BLOCK, k, l);
}

/* ------------------------------------------------------------------------ */
/* Matrix-vector and small-batch products                                    */
/* ------------------------------------------------------------------------ */

/* out[r] = dot(row r, (q, d)) for r < rows.  blocks: rows*(n/128) blocks. */
void q1o_gemv(const uint8_t *blocks, int64_t rows, int64_t n, const int8_t *q,
              const uint16_t *d, float *out)
{
    int64_t nb = n / Q1O_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        out[r] = q1o_dot_row(blocks + r * nb * Q1O_BLOCK_BYTES, nb, q, d);
}

/* Batched product: out[v*rows + r] = dot(row r, vector v), v < nvec.
 * q: nvec*n int8, d: nvec*(n/32) fp16.  Defined as the matrix-vector product
 * per vector (each row's lanes are independent chains). */
void q1o_gemm(const uint8_t *blocks, int64_t rows, int64_t n, int64_t nvec,
              const int8_t *q, const uint16_t *d, float *out)
{
    for (int64_t v = 0; v < nvec; ++v)
        q1o_gemv(blocks, rows, n, q + v * n, d + v * (n / Q1O_QBLOCK), out + v * rows);
}

/* Rows listed in `idx` only: out[i] = dot(row idx[i], vector vec_of[i]).
 * Used to check sampled outputs of full-size products one by one. */
void q1o_rows_sampled(const uint8_t *blocks, int64_t n, int64_t count,
                      const int64_t *idx, const int64_t *vec_of,
                      const int8_t *q, const uint16_t *d, float *out)
{
    int64_t nb = n / Q1O_BLOCK;
    for (int64_t i = 0; i < count; ++i) {
        int64_t v = vec_of ? vec_of[i] : 0;
        out[i] = q1o_dot_row(blocks + idx[i] * nb * Q1O_BLOCK_BYTES, nb,
                             q + v * n, d + v * (n / Q1O_QBLOCK));
    }
}

/* ------------------------------------------------------------------------ */
/* Q2_0 (ternary) weights                                                    */
/* ------------------------------------------------------------------------ */
/* The pages name a ternary sibling format, Q2_0, as the next GPU kernel
 * ("Advantages and efficiency", where optimization goes next; "Limitations":
 * no Q2_0 GPU kernel yet) and give its size only as 2.13 GB per 8B token
 * (par.md, benchmarks).  What it is here:
 *   OPEN-10 block = 2-byte little-endian fp16 scale d0, then 32 bytes of
 *           2-bit codes; element j's code is (qs[j>>2] >> 2*(j&3)) & 3 and its
 *           value t = code - 1, so 0, 1, 2 mean -1, 0, +1 (code 3 is not a
 *           weight); weight = t*d0.  34 bytes per 128 weights.
 *   OPEN-11 the row product is the Q1_0 chain with the lane sum taken over
 *           ternary values: +1 contributes q, -1 the wrapped negation of q,
 *           0 nothing.  Blocks, sub-blocks, lanes, the fma chain, the
 *           starting +0 and the horizontal sum are those of Q1_0 above. */
#define Q2O_BLOCK_BYTES 34

static int q2o_code(const uint8_t *blk, int j)
{
    return (blk[2 + (j >> 2)] >> (2 * (j & 3))) & 3;
}

/* Dequantized weight (row r, column j) of a rows x n Q2_0 matrix; NaN for
 * code 3. */
float q2o_weight(const uint8_t *blocks, int64_t n, int64_t r, int64_t j)
{
    const uint8_t *blk = blocks + (r * (n / Q1O_BLOCK) + j / Q1O_BLOCK) * Q2O_BLOCK_BYTES;
    int c = q2o_code(blk, (int)(j % Q1O_BLOCK));
    if (c == 3)
        return NAN;
    float d0 = q1o_f16_to_f32(q1o_block_scale_bits(blk));
    return (float)(c - 1) * d0;
}

/* Exact integer lane sum of sub-block k, lane l (OPEN-5, OPEN-11). */
static int32_t q2o_lane_sum(const uint8_t *blk, const int8_t *qb, int k, int l)
{
    int32_t s = 0;
    for (int i = 0; i < 4; ++i) {
        int j = Q1O_QBLOCK * k + 4 * l + i;
        int c = q2o_code(blk, j);
        if (c == 2)
            s += qb[j];
        else if (c == 0)
            s += q1o_neg_i8(qb[j]);
    }
    return s;
}

/* One output row of a Q2_0 matrix: nb 34-byte blocks against (q, d). */
float q2o_dot_row(const uint8_t *row_blocks, int64_t nb, const int8_t *q, const uint16_t *d)
{
    float acc[Q1O_LANES];
    for (int l = 0; l < Q1O_LANES; ++l)
        acc[l] = 0.0f;                                   /* OPEN-4 */
    for (int64_t b = 0; b < nb; ++b) {                   /* blocks in order */
        const uint8_t *blk = row_blocks + b * Q2O_BLOCK_BYTES;
        const int8_t *qb = q + b * Q1O_BLOCK;
        float d0 = q1o_f16_to_f32(q1o_block_scale_bits(blk));
        for (int l = 0; l < Q1O_LANES; ++l) {
            float ab = 0.0f;
            for (int k = 0; k < 4; ++k) {
                float d1 = q1o_f16_to_f32(d[b * 4 + k]);
                float t = (float)q2o_lane_sum(blk, qb, k, l);  /* exact: |s| <= 512 */
                ab = (k == 0) ? d1 * t : fmaf(d1, t, ab);
            }
            acc[l] = fmaf(d0, ab, acc[l]);
        }
    }
    return ((acc[0] + acc[4]) + (acc[2] + acc[6])) + ((acc[1] + acc[5]) + (acc[3] + acc[7]));
}

/* Exact integer lane sums s[b][k][l] of one Q2_0 row. */
void q2o_lane_sums(const uint8_t *row_blocks, int64_t nb, const int8_t *q, int32_t *s_out)
{
    for (int64_t b = 0; b < nb; ++b)
        for (int k = 0; k < 4; ++k)
            for (int l = 0; l < Q1O_LANES; ++l)
                s_out[(b * 4 + k) * Q1O_LANES + l] =
                    q2o_lane_sum(row_blocks + b * Q2O_BLOCK_BYTES, q + b * Q1O_BLOCK, k, l);
}

/* out[r] = dot(row r, (q, d)) for every row of a rows x n Q2_0 matrix. */
void q2o_gemv(const uint8_t *blocks, int64_t rows, int64_t n, const int8_t *q,
              const uint16_t *d, float *out)
{
    int64_t nb = n / Q1O_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        out[r] = q2o_dot_row(blocks + r * nb * Q2O_BLOCK_BYTES, nb, q, d);
}

/* Rows listed in `idx` only: out[i] = dot(row idx[i], (q, d)). */
void q2o_rows_sampled(const uint8_t *blocks, int64_t n, int64_t count, const int64_t *idx,
                      const int8_t *q, const uint16_t *d, float *out)
{
    int64_t nb = n / Q1O_BLOCK;
    for (int64_t i = 0; i < count; ++i)
        out[i] = q2o_dot_row(blocks + idx[i] * nb * Q2O_BLOCK_BYTES, nb, q, d);
}

/* ------------------------------------------------------------------------ */
/* Threaded oracle: rows claimed in 16-row chunks from an atomic counter      */
/* (bankML "docs/modules/par.md", "Technical usage": CHUNK_ROWS = 16, chunks  */
/* handed out dynamically; every row computed by the same single-thread      */
/* function, so the bits do not depend on the thread count).                 */
/* ------------------------------------------------------------------------ */

typedef float (*q1o_row_fn)(const uint8_t *, int64_t, const int8_t *, const uint16_t *);

typedef struct {
    q1o_row_fn row;          /* q1o_dot_row or q2o_dot_row                  */
    const uint8_t *blocks;
    int64_t rows, n, nb, nvec, block_bytes;
    const int8_t *q;         /* nvec * n quants                             */
    const uint16_t *d;       /* nvec * n/32 scales                          */
    float *out;              /* nvec * rows: out[v*rows + r]                */
    atomic_llong next;
    atomic_llong rows_done;
} q1o_job;

/* A claim is 16 consecutive rows; the claimant computes them for every
 * vector, each output by the single-thread row function. */
static void *q1o_worker(void *arg)
{
    q1o_job *job = (q1o_job *)arg;
    for (;;) {
        long long r0 = atomic_fetch_add(&job->next, Q1O_CHUNK_ROWS);
        if (r0 >= job->rows)
            break;
        long long r1 = r0 + Q1O_CHUNK_ROWS;
        if (r1 > job->rows)
            r1 = job->rows;
        for (int64_t v = 0; v < job->nvec; ++v)
            for (long long r = r0; r < r1; ++r)
                job->out[v * job->rows + r] =
                    job->row(job->blocks + r * job->nb * job->block_bytes, job->nb,
                             job->q + v * job->n, job->d + v * (job->n / Q1O_QBLOCK));
        atomic_fetch_add(&job->rows_done, r1 - r0);
    }
    return NULL;
}

/* Runs `job` on `threads` threads (the calling thread is worker 0).  Returns
 * the number of rows written (== rows on success), or -1 if a thread could
 * not be started. */
static long long q1o_run_threaded(q1o_job *job, int threads)
{
    if (threads < 1)
        threads = 1;
    atomic_init(&job->next, 0);
    atomic_init(&job->rows_done, 0);
    pthread_t *tid = NULL;
    int started = 0;
    if (threads > 1) {
        tid = (pthread_t *)calloc((size_t)threads - 1, sizeof(pthread_t));
        if (!tid)
            return -1;
        for (int t = 0; t < threads - 1; ++t) {
            if (pthread_create(&tid[t], NULL, q1o_worker, job) != 0)
                break;
            ++started;
        }
    }
    q1o_worker(job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    if (threads > 1 && started != threads - 1)
        return -1;
    return (long long)atomic_load(&job->rows_done);
}

static long long q1o_threaded(q1o_row_fn row, int64_t block_bytes, const uint8_t *blocks, int64_t rows,
                              int64_t n, int64_t nvec, const int8_t *q, const uint16_t *d, float *out,
                              int threads)
{
    q1o_job job;
    job.row = row;
    job.blocks = blocks;
    job.rows = rows;
    job.n = n;
    job.nb = n / Q1O_BLOCK;
    job.nvec = nvec;
    job.block_bytes = block_bytes;
    job.q = q;
    job.d = d;
    job.out = out;
    return q1o_run_threaded(&job, threads);
}

/* Matrix-vector product on `threads` threads: out[r] = q1o_dot_row(row r). */
long long q1o_gemv_threaded(const uint8_t *blocks, int64_t rows, int64_t n,
                            const int8_t *q, const uint16_t *d, float *out, int threads)
{
    return q1o_threaded(q1o_dot_row, Q1O_BLOCK_BYTES, blocks, rows, n, 1, q, d, out, threads);
}

/* Batched product on `threads` threads: out[v*rows + r] as q1o_gemm. */
long long q1o_gemm_threaded(const uint8_t *blocks, int64_t rows, int64_t n, int64_t nvec,
                            const int8_t *q, const uint16_t *d, float *out, int threads)
{
    return q1o_threaded(q1o_dot_row, Q1O_BLOCK_BYTES, blocks, rows, n, nvec, q, d, out, threads);
}

/* Q2_0 matrix-vector product on `threads` threads: out[r] = q2o_dot_row(row r). */
long long q2o_gemv_threaded(const uint8_t *blocks, int64_t rows, int64_t n,
                            const int8_t *q, const uint16_t *d, float *out, int threads)
{
    return q1o_threaded(q2o_dot_row, Q2O_BLOCK_BYTES, blocks, rows, n, 1, q, d, out, threads);
}
