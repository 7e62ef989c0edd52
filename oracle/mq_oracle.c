/*
 * mq_oracle.c -- the oracle: a plain, slow, single-threaded CPU statement of
 * what the k-quant batch-1 decode GEMV ("MMVQ") and its q8 producers compute.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs load this file.  The library
 * (include/mq.h, quant_quantized_gemv_gb300/csrc) never calls it, shares no
 * header, table or helper with it, and the oracle knows nothing of the
 * library's repacked layout: it always reads weights in the GGUF block order.
 *
 * Sources ("the pages" = the minfer engineering log, cited by page and
 * section):
 *   [D4-4] "76 · D4-4 — dpl dense split-plane q6_K decode MMVQ lands"
 *   [D4-2] "74 · D4-2 — B0 latent correctness fix"
 *   [D3]   "67 · D3: 14B decode attribution + the D3b bitwise MMVQ triple"
 *   [D3-5] "70 · D3-5 — fused-producer decode A-quantize"
 *   [D3a]  "68 · D3a fattn rewrite" (tolerance calibration only)
 *
 * Precision: floating point is fp64 except where the pages fix it.  The pages
 * fix the q8 quantizer in f32 ([D3-5] §3.2, the shared per-32-block body), so
 * mqo_quantize_q8 runs in f32 exactly as printed there.  The dot products are
 * integer (exact) and the scale combine is fp64, where every term
 * f16 * int6 * int * f16 is exact (fewer than 53 significant bits).
 *
 * Parity pins for every function are in tests/test_oracle_pins.py.  The q4_K
 * block format is not on the pages; it follows the GGUF q4_K field list
 * (fp16 d, fp16 dmin, 12 bytes of packed 6-bit scales/mins, 128 bytes of
 * nibbles) and is pinned by hand-built blocks with closed-form values.
 * q5_K is only named on the pages (a sibling MMVQ class, [D3-5] §4); its
 * block is GGUF q5_K: the q4_K fields plus 32 bytes holding each weight's
 * fifth bit, pinned the same way.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math, so
 * that IEEE division, rintf and the f16 rounding below are the ones C defines).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define QK 256          /* weights per k-quant super-block                   */
#define Q6K_BYTES 210   /* [D4-4] §1: ql 128 + qh 64 + sc 16 + d 2            */
#define Q4K_BYTES 144   /* GGUF q4_K: d 2 + dmin 2 + scales 12 + qs 128       */
#define Q5K_BYTES 176   /* GGUF q5_K: d 2 + dmin 2 + scales 12 + qh 32 + qs 128 */
#define Q8_BLOCK 32     /* [D3-5] §3.2: q8 activation blocks of 32 values     */

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32.  f16 -> f32 is exact; f32 -> f16 rounds to    */
/* nearest-even (the behaviour of __float2half in [D3-5] §3.2), subnormals   */
/* included.  Written from the IEEE 754 encoding, not from any CUDA header.  */
/* ------------------------------------------------------------------------ */
float mqo_f16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int ex = (h >> 10) & 0x1f;
    const int man = h & 0x3ff;
    float v;
    if (ex == 0)
        v = ldexpf((float)man, -24);                 /* zero or subnormal     */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexpf((float)(man | 0x400), ex - 25);   /* 1.man * 2^(ex-15)     */
    return sign ? -v : v;
}

uint16_t mqo_f32_to_f16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, 4);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    const float a = fabsf(f);
    if (a >= 65520.0f)                 /* halfway past 65504 rounds up to inf */
        return (uint16_t)(sign | 0x7c00u);
    if (a < 6.103515625e-05f) {        /* below 2^-14: subnormal (or zero)    */
        /* a * 2^24 is exact in f32; rintf rounds half to even.  A result of
         * 1024 is the smallest normal, whose encoding is also 1024.         */
        const float m = rintf(ldexpf(a, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e2;
    (void)frexpf(a, &e2);              /* a = fr * 2^e2, fr in [0.5, 1)       */
    const int e = e2 - 1;              /* a = 1.x * 2^e, e in [-14, 15]       */
    const float m = rintf(ldexpf(a, 10 - e));   /* exact scale, then RNE      */
    /* m in [1024, 2048]; m == 2048 carries into the exponent field.          */
    const uint32_t h = ((uint32_t)(e + 15) << 10) + ((uint32_t)m - 1024u);
    return (uint16_t)(sign | h);
}

/* ------------------------------------------------------------------------ */
/* q8 activation quantizer, one 32-value block ([D3-5] §3.2, the shared      */
/* per-32-block body; §2.3 for why the bytes are a per-element function).   */
/*   am = max |x_i| (fmaxf chain from 0)                                     */
/*   d  = am / 127 (f32 division)                                            */
/*   di = d != 0 ? 1/d : 0 (f32 reciprocal, then a multiply)                 */
/*   q_i = clamp(rint(x_i * di), -128, 127)  (rint: round half to even)      */
/*   stored: dh = f16(d), the 32 q_i, sum = sum of q_i (int32)               */
/* ------------------------------------------------------------------------ */
void mqo_quantize_q8(const float *x, int n, uint16_t *d_out, int8_t *q_out,
                     int32_t *sum_out)
{
    for (int b = 0; b < n / Q8_BLOCK; ++b) {
        const float *xb = x + (size_t)b * Q8_BLOCK;
        float am = 0.0f;
        for (int i = 0; i < Q8_BLOCK; ++i)
            am = fmaxf(am, fabsf(xb[i]));
        const float d = am / 127.0f;
        const float di = (d != 0.0f) ? 1.0f / d : 0.0f;
        d_out[b] = mqo_f32_to_f16(d);
        int32_t s = 0;
        for (int i = 0; i < Q8_BLOCK; ++i) {
            const float p = xb[i] * di;
            int q = (int)rintf(p);
            if (q < -128) q = -128;
            if (q > 127) q = 127;
            q_out[(size_t)b * Q8_BLOCK + i] = (int8_t)q;
            s += q;
        }
        sum_out[b] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* q6_K element decode.  A super-block holds 256 weights as                  */
/*   ql[128] @0 (low 4 bits), qh[64] @128 (high 2 bits), sc[16] @192 (int8   */
/*   sub-block scales), d @208 (fp16)            -- [D4-4] §1, §2;           */
/* the is-pair ("unit") addressing of [D4-4] §3.2 Excerpt B and [D4-2] §3.2  */
/* Excerpt C: unit u of a block is pair p = 0..7, half = p >> 2, g = p & 3;  */
/* its ql bytes start at half*64 + (g&1)*32, its qh bytes at half*32 with    */
/* bit shift 2g, and its two scales are sc[2p] and sc[2p+1].  Element        */
/* e = 32p + l (l = 0..31) therefore reads the low nibble (g < 2) or the     */
/* high nibble (g >= 2) of ql[half*64 + (g&1)*32 + l] and bits 2g..2g+1 of   */
/* qh[half*32 + l]; q = (lo | hi << 4) - 32 (the GGUF offset, which the      */
/* pages elide).  Sub-block s = 2p + (l >= 16) = e / 16.                     */
/* ------------------------------------------------------------------------ */
static int q6k_q(const uint8_t *blk, int e)
{
    const int p = e >> 5, l = e & 31;
    const int half = p >> 2, g = p & 3;
    const int qlb = blk[half * 64 + (g & 1) * 32 + l];
    const int lo = (g < 2) ? (qlb & 0x0f) : (qlb >> 4);
    const int hi = (blk[128 + half * 32 + l] >> (2 * g)) & 3;
    return (lo | (hi << 4)) - 32;
}

static int q6k_scale(const uint8_t *blk, int s) { return (int)(int8_t)blk[192 + s]; }

static double q6k_d(const uint8_t *blk)
{
    return (double)mqo_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8)));
}

/* Dequantize nblocks q6_K blocks to fp64: w_e = f16(d) * sc[e/16] * q_e. */
void mqo_dequant_q6k(const uint8_t *blocks, long nblocks, double *w)
{
    for (long b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + (size_t)b * Q6K_BYTES;
        const double d = q6k_d(blk);
        for (int e = 0; e < QK; ++e)
            w[(size_t)b * QK + e] = d * (double)q6k_scale(blk, e >> 4) * (double)q6k_q(blk, e);
    }
}

/* ------------------------------------------------------------------------ */
/* q4_K element decode (GGUF q4_K; not on the pages).  Block: d (fp16) @0,   */
/* dmin (fp16) @2, scales[12] @4, qs[128] @16.  Sub-block k = 0..7 holds 32  */
/* weights; element e = 32k + l is the low nibble (k even) or high nibble    */
/* (k odd) of qs[32*(k/2) + l].  The 6-bit scale sc_k and min m_k:           */
/*   k < 4:  sc = scales[k] & 63,  m = scales[k+4] & 63                      */
/*   k >= 4: sc = (scales[k+4] & 15) | (scales[k-4] >> 6) << 4               */
/*           m  = (scales[k+4] >> 4) | (scales[k]   >> 6) << 4               */
/* and w_e = f16(d) * sc_k * q_e - f16(dmin) * m_k.                          */
/* ------------------------------------------------------------------------ */
static int q4k_q(const uint8_t *blk, int e)
{
    const int k = e >> 5, l = e & 31;
    const int byte = blk[16 + 32 * (k >> 1) + l];
    return (k & 1) ? (byte >> 4) : (byte & 0x0f);
}

void mqo_q4k_scale_min(const uint8_t *blk, int k, int *sc, int *m)
{
    const uint8_t *s = blk + 4;
    if (k < 4) {
        *sc = s[k] & 63;
        *m = s[k + 4] & 63;
    } else {
        *sc = (s[k + 4] & 15) | ((s[k - 4] >> 6) << 4);
        *m = (s[k + 4] >> 4) | ((s[k] >> 6) << 4);
    }
}

static double q4k_half(const uint8_t *blk, int off)
{
    return (double)mqo_f16_to_f32((uint16_t)(blk[off] | (blk[off + 1] << 8)));
}

void mqo_dequant_q4k(const uint8_t *blocks, long nblocks, double *w)
{
    for (long b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + (size_t)b * Q4K_BYTES;
        const double d = q4k_half(blk, 0), dmin = q4k_half(blk, 2);
        for (int e = 0; e < QK; ++e) {
            int sc, m;
            mqo_q4k_scale_min(blk, e >> 5, &sc, &m);
            w[(size_t)b * QK + e] = d * (double)sc * (double)q4k_q(blk, e) - dmin * (double)m;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* q5_K element decode (GGUF q5_K; named but not printed on the pages).      */
/* Block: d (fp16) @0, dmin (fp16) @2, scales[12] @4 (packed exactly as in   */
/* q4_K), qh[32] @16, qs[128] @48.  Element e = 32k + l of sub-block k takes */
/* its low 4 bits from qs as q4_K does (low nibble of qs[32*(k/2) + l] for k */
/* even, high nibble for k odd) and its fifth bit from bit k of qh[l]:       */
/*   q_e = nibble + 16 * ((qh[l] >> k) & 1),  0 <= q_e <= 31,                */
/*   w_e = f16(d) * sc_k * q_e - f16(dmin) * m_k.                            */
/* ------------------------------------------------------------------------ */
static int q5k_q(const uint8_t *blk, int e)
{
    const int k = e >> 5, l = e & 31;
    const int byte = blk[48 + 32 * (k >> 1) + l];
    const int lo = (k & 1) ? (byte >> 4) : (byte & 0x0f);
    return lo + 16 * ((blk[16 + l] >> k) & 1);
}

void mqo_dequant_q5k(const uint8_t *blocks, long nblocks, double *w)
{
    for (long b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + (size_t)b * Q5K_BYTES;
        const double d = q4k_half(blk, 0), dmin = q4k_half(blk, 2);
        for (int e = 0; e < QK; ++e) {
            int sc, m;
            mqo_q4k_scale_min(blk, e >> 5, &sc, &m);
            w[(size_t)b * QK + e] = d * (double)sc * (double)q5k_q(blk, e) - dmin * (double)m;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Integer sub-block dots (the bit-exact intermediate).                     */
/*   q6_K: isum_s = sum over the 16 weights of sub-block s of (q-32)*q8      */
/*         ([D4-2] §3.2 Excerpt C: one dp4a tree per 16-weight sub-block).   */
/*   q4_K, q5_K: isum_k = sum over the 32 weights of sub-block k of q*q8.    */
/* W is GGUF-ordered, rows x (cols/256) blocks; q8 holds cols int8 values.   */
/* Output: rows x nb x 16 (q6_K) or rows x nb x 8 (q4_K, q5_K) int32.        */
/* ------------------------------------------------------------------------ */
void mqo_subdots_q6k(const uint8_t *W, const int8_t *q8, int rows, int cols, int32_t *isums)
{
    const int nb = cols / QK;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q6K_BYTES;
            for (int s = 0; s < 16; ++s) {
                int32_t acc = 0;
                for (int e = 16 * s; e < 16 * s + 16; ++e)
                    acc += q6k_q(blk, e) * (int32_t)q8[(size_t)b * QK + e];
                isums[((size_t)r * nb + b) * 16 + s] = acc;
            }
        }
}

void mqo_subdots_q4k(const uint8_t *W, const int8_t *q8, int rows, int cols, int32_t *isums)
{
    const int nb = cols / QK;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q4K_BYTES;
            for (int k = 0; k < 8; ++k) {
                int32_t acc = 0;
                for (int e = 32 * k; e < 32 * k + 32; ++e)
                    acc += q4k_q(blk, e) * (int32_t)q8[(size_t)b * QK + e];
                isums[((size_t)r * nb + b) * 8 + k] = acc;
            }
        }
}

void mqo_subdots_q5k(const uint8_t *W, const int8_t *q8, int rows, int cols, int32_t *isums)
{
    const int nb = cols / QK;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q5K_BYTES;
            for (int k = 0; k < 8; ++k) {
                int32_t acc = 0;
                for (int e = 32 * k; e < 32 * k + 32; ++e)
                    acc += q5k_q(blk, e) * (int32_t)q8[(size_t)b * QK + e];
                isums[((size_t)r * nb + b) * 8 + k] = acc;
            }
        }
}

/* ------------------------------------------------------------------------ */
/* GEMV y = W x_hat, x_hat_i = f16(d8_{i/32}) * q8_i.                        */
/* q6_K ([D4-2] §3.2 Excerpt C, the per-unit accumulation statement):        */
/*   y_r = sum_b sum_s f16(d_b) * sc_s * f16(d8_{u(s)}) * isum_s             */
/* q4_K, q5_K (the GGUF decode multiplied out against x_hat):               */
/*   y_r = sum_b sum_k f16(d8_k) * (f16(d)*sc_k*isum_k - f16(dmin)*m_k*qsum_k)*/
/*   with qsum_k = sum of the q8 values of block k.                          */
/* Accumulated in fp64 in ascending (b, s); absum receives sum |term| per    */
/* row, the scale of the float tolerance.  Row range [r0, r1) so that        */
/* callers can split the rows over host threads.                             */
/* ------------------------------------------------------------------------ */
void mqo_gemv_q6k(const uint8_t *W, const uint16_t *d8, const int8_t *q8,
                  int r0, int r1, int cols, double *y, double *absum)
{
    const int nb = cols / QK;
    for (int r = r0; r < r1; ++r) {
        double acc = 0.0, aacc = 0.0;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q6K_BYTES;
            const double d = q6k_d(blk);
            for (int s = 0; s < 16; ++s) {
                int32_t isum = 0;
                for (int e = 16 * s; e < 16 * s + 16; ++e)
                    isum += q6k_q(blk, e) * (int32_t)q8[(size_t)b * QK + e];
                const double d8v = (double)mqo_f16_to_f32(d8[(size_t)b * 8 + s / 2]);
                const double term = d * (double)q6k_scale(blk, s) * d8v * (double)isum;
                acc += term;
                aacc += fabs(term);
            }
        }
        y[r] = acc;
        if (absum) absum[r] = aacc;
    }
}

void mqo_gemv_q4k(const uint8_t *W, const uint16_t *d8, const int8_t *q8,
                  int r0, int r1, int cols, double *y, double *absum)
{
    const int nb = cols / QK;
    for (int r = r0; r < r1; ++r) {
        double acc = 0.0, aacc = 0.0;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q4K_BYTES;
            const double d = q4k_half(blk, 0), dmin = q4k_half(blk, 2);
            for (int k = 0; k < 8; ++k) {
                int sc, m;
                mqo_q4k_scale_min(blk, k, &sc, &m);
                int32_t isum = 0, qsum = 0;
                for (int e = 32 * k; e < 32 * k + 32; ++e) {
                    const int32_t xv = q8[(size_t)b * QK + e];
                    isum += q4k_q(blk, e) * xv;
                    qsum += xv;
                }
                const double d8v = (double)mqo_f16_to_f32(d8[(size_t)b * 8 + k]);
                const double t1 = d8v * d * (double)sc * (double)isum;
                const double t2 = d8v * dmin * (double)m * (double)qsum;
                acc += t1 - t2;
                aacc += fabs(t1) + fabs(t2);
            }
        }
        y[r] = acc;
        if (absum) absum[r] = aacc;
    }
}

void mqo_gemv_q5k(const uint8_t *W, const uint16_t *d8, const int8_t *q8,
                  int r0, int r1, int cols, double *y, double *absum)
{
    const int nb = cols / QK;
    for (int r = r0; r < r1; ++r) {
        double acc = 0.0, aacc = 0.0;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q5K_BYTES;
            const double d = q4k_half(blk, 0), dmin = q4k_half(blk, 2);
            for (int k = 0; k < 8; ++k) {
                int sc, m;
                mqo_q4k_scale_min(blk, k, &sc, &m);
                int32_t isum = 0, qsum = 0;
                for (int e = 32 * k; e < 32 * k + 32; ++e) {
                    const int32_t xv = q8[(size_t)b * QK + e];
                    isum += q5k_q(blk, e) * xv;
                    qsum += xv;
                }
                const double d8v = (double)mqo_f16_to_f32(d8[(size_t)b * 8 + k]);
                const double t1 = d8v * d * (double)sc * (double)isum;
                const double t2 = d8v * dmin * (double)m * (double)qsum;
                acc += t1 - t2;
                aacc += fabs(t1) + fabs(t2);
            }
        }
        y[r] = acc;
        if (absum) absum[r] = aacc;
    }
}

/* ------------------------------------------------------------------------ */
/* The f32-activation q6_K GEMV ([D3] §2.3 and §3.3: the "padded f32"        */
/* family, which dequantizes each block and multiplies it into the f32       */
/* activation row directly, without a q8 producer):                          */
/*   y_r = sum_b sum_e w_{r,b,e} * x_{256b+e},  w = f16(d) * sc_{e/16} * q_e */
/* Every term is exact in fp64 (w has at most 11 + 7 + 6 significant bits,   */
/* x at most 24), summed in ascending (b, e); absum receives sum |term|.     */
/* ------------------------------------------------------------------------ */
void mqo_gemv_q6k_f32(const uint8_t *W, const float *x, int r0, int r1, int cols,
                      double *y, double *absum)
{
    const int nb = cols / QK;
    for (int r = r0; r < r1; ++r) {
        double acc = 0.0, aacc = 0.0;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = W + ((size_t)r * nb + b) * Q6K_BYTES;
            const double d = q6k_d(blk);
            for (int e = 0; e < QK; ++e) {
                const double w = d * (double)q6k_scale(blk, e >> 4) * (double)q6k_q(blk, e);
                const double term = w * (double)x[(size_t)b * QK + e];
                acc += term;
                aacc += fabs(term);
            }
        }
        y[r] = acc;
        if (absum) absum[r] = aacc;
    }
}

/* ------------------------------------------------------------------------ */
/* Producers ([D3-5] §3.2).  The rms body is not printed on the pages; the   */
/* plain reading is y_i = x_i / sqrt(mean(x^2) + eps) * gain_i.  SwiGLU is   */
/* printed: y_i = (g_i / (1 + exp(-g_i))) * u_i.  Both in fp64.              */
/* ------------------------------------------------------------------------ */
void mqo_rmsnorm(const float *x, const float *gain, float eps, int n, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += (double)x[i] * (double)x[i];
    const double scale = 1.0 / sqrt(ss / (double)n + (double)eps);
    for (int i = 0; i < n; ++i)
        y[i] = (double)x[i] * scale * (double)gain[i];
}

void mqo_swiglu(const float *g, const float *u, int n, double *y)
{
    for (int i = 0; i < n; ++i) {
        const double gv = (double)g[i];
        y[i] = (gv / (1.0 + exp(-gv))) * (double)u[i];
    }
}
