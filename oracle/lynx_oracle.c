/*
 * lynx_oracle.c -- plain, slow CPU oracle of the Lynx progressive KV quantizer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. It shares no code, header,
 * table or constant with the CUDA library; both sides build their tables from
 * the same written definitions.
 *
 * Source: "Lynx: the KV cache does not have to arrive whole" (aigenapps
 * reading of Han et al.), section 3 "The quantizer" and section 4
 * "Speculation at the communication boundary". Steps follow the page's order:
 *   stage 1  page-level normalisation, per channel, to [0,1]
 *   stage 2  chunk-wise outlier isolation, C = 32 tokens: centre by the local
 *            mean, divide by the local max-abs
 *   stage 3  alpha-law logarithmic map onto 2^7 - 1 = 127 levels, with the
 *            sign-aware mapping of small negatives
 *   stage 4  +7 round-half-down bias, then a 4-bit anchor / 4-bit residual cut
 * Where the page leaves a step open, the reading taken is written next to it.
 *
 * Numeric contract of the encoder (fp32, every operation rounded to nearest,
 * no fused multiply-add; build with -ffp-contract=off):
 *   mn = min x + 0, rng = (max x + 0) - mn (a zero extreme is +0),
 *   inv_r = rng > 0 ? 1/rng : 0, u = (x-mn)*inv_r
 *   chunk sum = stride-halving pairwise tree over 32 slots (+16, +8, +4, +2, +1),
 *   absent slots hold +0; mean = sum / n_c; mu = fp16 nearest(mean);
 *   v = u - mu; s = fp16 rounded up(max |v|); inv_s = s > 0 ? 1/s : 0; w = v*inv_s
 *   q = #{k in 1..63 : |w| >= T_k}, T_k = fp32(((1+alpha)^((k-1/2)/63) - 1)/alpha)
 *   c = q for w >= 0, c = -max(q,1) for w < 0
 *   b = c + 7, A = floor(b/16), r = b - 16A; stored nibbles A & 15 and r.
 * Statistics fp32 cannot carry (the pages are silent; reading taken here): a
 *   NaN among a channel's valid values makes its stored min and range the
 *   quiet NaN 0x7FC00000 (any NaN range is stored as that pattern); when the
 *   range or its reciprocal is not finite (a NaN or infinite value, a range
 *   beyond fp32, a subnormal range whose reciprocal overflows) every u of the
 *   channel is 0, so its chunk means and scales are 0 and its codes 0.
 * Decode (fp64 here): Lv[k] = fp16 nearest(((1+alpha)^(k/63) - 1)/alpha);
 *   anchor-only code 16A, full code 16A + r - 7;
 *   x = mn + rng * (mu + s * sgn(code) * Lv[min(|code|, 64)]).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_PAGE 256     /* tokens per page (section 3) */
#define ORC_CHUNK 32     /* C = 32 tokens per chunk (section 3) */
#define ORC_NCHUNK (ORC_PAGE / ORC_CHUNK)
#define ORC_D 128        /* head dimension of the worked example (section 1) */
#define ORC_QMAX 63      /* 127 levels = codes -63..63 (section 3) */
#define ORC_BIAS 7       /* round-half-down bias before the 4-bit shift (section 3) */
#define ORC_ALPHA 255.0  /* alpha of the alpha-law map; the page gives no value */

/* ------------------------------------------------------------------ */
/* number formats                                                     */
/* ------------------------------------------------------------------ */

static float qnan_f32(void)
{
    uint32_t b = 0x7FC00000u;
    float f;
    memcpy(&f, &b, 4);
    return f;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary16 bits of a finite double, rounded to nearest-even (up == 0) or
 * toward +infinity (up == 1). Written from the IEEE 754 binary16 format:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits, subnormal
 * quantum 2^-24, largest finite 65504. */
uint16_t orc_f16_from_double(double x, int up)
{
    uint16_t sign = 0;
    double v = x;
    if (signbit(x)) {
        sign = 0x8000;
        v = -x;
    }
    if (v == 0.0)
        return sign;
    int e2;
    frexp(v, &e2);            /* v = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;           /* 2^e <= v < 2^(e+1) */
    int qexp = (e < -14) ? -24 : e - 10;
    double n = ldexp(v, -qexp); /* exact: v has at most 53 bits */
    double nr;
    if (!up)
        nr = nearbyint(n);      /* ties to even in the default rounding mode */
    else
        nr = sign ? floor(n) : ceil(n);
    double r = ldexp(nr, qexp);
    if (r == 0.0)
        return sign;
    if (r > 65504.0)
        return (uint16_t)(sign | 0x7C00);
    frexp(r, &e2);
    e = e2 - 1;
    if (e < -14)
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    uint16_t frac = (uint16_t)(ldexp(r, 10 - e) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | frac);
}

double orc_f16_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* ------------------------------------------------------------------ */
/* tables (section 3, "Non-linear transform" and "The cut")           */
/* ------------------------------------------------------------------ */

double orc_alpha(void) { return ORC_ALPHA; }

/* thr[k], k = 1..63: fp32 value of the point where the alpha-law map
 * 63 * ln(1 + alpha y) / ln(1 + alpha) crosses k - 1/2; thr[0] = 0.
 * lv[k], k = 0..64: fp16 bits of the level value ((1+alpha)^(k/63) - 1)/alpha. */
void orc_tables(float *thr, uint16_t *lv)
{
    const double a = ORC_ALPHA;
    thr[0] = 0.0f;
    for (int k = 1; k <= ORC_QMAX; ++k)
        thr[k] = (float)((pow(1.0 + a, (k - 0.5) / ORC_QMAX) - 1.0) / a);
    for (int k = 0; k <= 64; ++k)
        lv[k] = orc_f16_from_double((pow(1.0 + a, (double)k / ORC_QMAX) - 1.0) / a, 0);
}

/* Stage 3 for one value: level count, then the sign-aware code.
 * Reading: the map rounds half up in the log domain (a threshold count), and a
 * negative w whose level rounds to 0 becomes -1 (the sign-aware rule), so a
 * small negative value decodes below the chunk mean; other negatives keep -q. */
static int code_of(float w, const float *thr)
{
    float a = fabsf(w);
    int q = 0;
    for (int k = 1; k <= ORC_QMAX; ++k)
        if (a >= thr[k])
            ++q;
    if (w < 0.0f)
        return -(q > 1 ? q : 1);
    return q;
}

void orc_codes(const float *w, int64_t n, int8_t *codes)
{
    float thr[64];
    uint16_t lv[65];
    orc_tables(thr, lv);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        codes[i] = (int8_t)code_of(w[i], thr);
}

/* Stage 4: +7 then the 4-bit cut. A = floor((c+7)/16) in [-4, 4], r in [0, 15]. */
static void split_code(int c, int *A, int *r)
{
    int b = c + ORC_BIAS;
    int rr = ((b % 16) + 16) % 16;
    *A = (b - rr) / 16;
    *r = rr;
}

void orc_split(const int8_t *codes, int64_t n, int8_t *A, uint8_t *r)
{
    for (int64_t i = 0; i < n; ++i) {
        int a, rr;
        split_code(codes[i], &a, &rr);
        A[i] = (int8_t)a;
        r[i] = (uint8_t)rr;
    }
}

/* ------------------------------------------------------------------ */
/* encoder, one page                                                  */
/* ------------------------------------------------------------------ */

/* x: 256 rows of 128 bf16 values (row = token), of which the first n are
 * valid. Outputs, for this page only:
 *   anc, res   256 rows x 64 bytes; byte d/2 holds channel d (even d in the low nibble)
 *   pm         [2][128] fp32: page minimum, page range
 *   cm         [8][2][128] fp16 bits: chunk mean, chunk scale              */
static void encode_page(const uint16_t *x, int n, const float *thr, uint8_t *anc, uint8_t *res,
                        float *pm, uint16_t *cm)
{
    float u[ORC_PAGE];
    int8_t codes[ORC_PAGE][ORC_D];
    memset(codes, 0, sizeof codes); /* tokens past n keep code 0 */

    for (int d = 0; d < ORC_D; ++d) {
        /* stage 1: page-level normalisation over the valid tokens */
        float mn = 0.0f, rng = 0.0f;
        if (n > 0) {
            float mx = -INFINITY;
            int has_nan = 0;
            mn = INFINITY;
            for (int t = 0; t < n; ++t) {
                float v = bf16_to_f32(x[(size_t)t * ORC_D + d]);
                if (v != v) {
                    has_nan = 1;
                    continue;
                }
                if (v < mn)
                    mn = v;
                if (v > mx)
                    mx = v;
            }
            /* a zero extreme is +0 whichever zero the data held, so that the
             * metadata bits do not depend on the order of the scan */
            mn = mn + 0.0f;
            mx = mx + 0.0f;
            rng = mx - mn;
            if (has_nan)
                mn = rng = qnan_f32();
            if (rng != rng)
                rng = qnan_f32();
        }
        float inv_r = rng > 0.0f ? 1.0f / rng : 0.0f;
        /* statistics fp32 cannot carry: the channel is coded as constant */
        int degenerate = !(rng <= FLT_MAX) || !(inv_r <= FLT_MAX);
        for (int t = 0; t < n; ++t)
            u[t] = degenerate ? 0.0f : (bf16_to_f32(x[(size_t)t * ORC_D + d]) - mn) * inv_r;
        pm[d] = mn;
        pm[ORC_D + d] = rng;

        /* stage 2: chunk-wise isolation, C = 32 */
        for (int j = 0; j < ORC_NCHUNK; ++j) {
            int nc = n - j * ORC_CHUNK;
            if (nc > ORC_CHUNK)
                nc = ORC_CHUNK;
            uint16_t mu_h = 0, s_h = 0;
            if (nc > 0) {
                float slot[ORC_CHUNK];
                for (int i = 0; i < ORC_CHUNK; ++i)
                    slot[i] = i < nc ? u[j * ORC_CHUNK + i] : 0.0f;
                for (int h = ORC_CHUNK / 2; h >= 1; h /= 2)
                    for (int i = 0; i < h; ++i)
                        slot[i] = slot[i] + slot[i + h];
                float mean = slot[0] / (float)nc;
                mu_h = orc_f16_from_double((double)mean, 0);
                float mu = (float)orc_f16_to_double(mu_h);
                float s = 0.0f;
                for (int i = 0; i < nc; ++i) {
                    float v = u[j * ORC_CHUNK + i] - mu;
                    float av = fabsf(v);
                    if (av > s)
                        s = av;
                }
                s_h = orc_f16_from_double((double)s, 1);
                float sf = (float)orc_f16_to_double(s_h);
                float inv_s = sf > 0.0f ? 1.0f / sf : 0.0f;
                /* stage 3: alpha-law map with sign-aware mapping */
                for (int i = 0; i < nc; ++i) {
                    float v = u[j * ORC_CHUNK + i] - mu;
                    float w = v * inv_s;
                    codes[j * ORC_CHUNK + i][d] = (int8_t)code_of(w, thr);
                }
            }
            cm[(j * 2 + 0) * ORC_D + d] = mu_h;
            cm[(j * 2 + 1) * ORC_D + d] = s_h;
        }
    }

    /* stage 4: bias, cut and nibble packing */
    for (int t = 0; t < ORC_PAGE; ++t) {
        for (int d = 0; d < ORC_D; d += 2) {
            int a0, r0, a1, r1;
            split_code(codes[t][d], &a0, &r0);
            split_code(codes[t][d + 1], &a1, &r1);
            anc[t * (ORC_D / 2) + d / 2] = (uint8_t)(((unsigned)a0 & 15u) | (((unsigned)a1 & 15u) << 4));
            res[t * (ORC_D / 2) + d / 2] = (uint8_t)((unsigned)r0 | ((unsigned)r1 << 4));
        }
    }
}

/* x: [L][H][T][128] bf16 bits, T a multiple of 256. page_valid: [T/256]
 * valid-token counts (0..256) shared by every (layer, head), or NULL for
 * full pages. Outputs use the library's layout:
 *   anc, res  [L][H][T][64]; pm [L][H][T/256][2][128]; cm [L][H][T/256][8][2][128]. */
int orc_quantize(const uint16_t *x, int L, int H, int T, const int32_t *page_valid, uint8_t *anc,
                 uint8_t *res, float *pm, uint16_t *cm)
{
    if (L < 0 || H < 0 || T < 0 || T % ORC_PAGE)
        return 1;
    float thr[64];
    uint16_t lv[65];
    orc_tables(thr, lv);
    const int P = T / ORC_PAGE;
    const int64_t units = (int64_t)L * H * P;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t id = 0; id < units; ++id) {
        int p = (int)(id % P);
        int64_t lh = id / P;
        int n = page_valid ? page_valid[p] : ORC_PAGE;
        if (n < 0)
            n = 0;
        if (n > ORC_PAGE)
            n = ORC_PAGE;
        size_t row0 = (size_t)lh * T + (size_t)p * ORC_PAGE;
        encode_page(x + row0 * ORC_D, n, thr, anc + row0 * (ORC_D / 2), res + row0 * (ORC_D / 2),
                    pm + (size_t)id * 2 * ORC_D, cm + (size_t)id * ORC_NCHUNK * 2 * ORC_D);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* decoders (section 3 "The cut", section 4)                          */
/* ------------------------------------------------------------------ */

static int nib_signed(unsigned v) { return v >= 8 ? (int)v - 16 : (int)v; }

/* Value of the code of channel d of row `row` (a row of the [T][128] view of
 * one (layer, head)); `full` selects anchor+residual, else anchor alone with
 * the residual taken at its centre. Codes outside -64..64 can only come from
 * planes the encoder did not write; their magnitude saturates at Lv[64]. */
static double decode_one(const uint8_t *anc, const uint8_t *res, const float *pm,
                         const uint16_t *cm, const double *lvd, size_t row, int d, int full)
{
    size_t p = row / ORC_PAGE;
    int j = (int)((row % ORC_PAGE) / ORC_CHUNK);
    unsigned ab = anc[row * (ORC_D / 2) + d / 2];
    int A = nib_signed((d & 1) ? (ab >> 4) : (ab & 15u));
    int c = 16 * A;
    if (full) {
        unsigned rb = res[row * (ORC_D / 2) + d / 2];
        int r = (int)((d & 1) ? (rb >> 4) : (rb & 15u));
        c = 16 * A + r - ORC_BIAS;
    }
    int k = c < 0 ? -c : c;
    if (k > 64)
        k = 64;
    double sg = c > 0 ? 1.0 : (c < 0 ? -1.0 : 0.0);
    double mn = pm[p * 2 * ORC_D + d];
    double rng = pm[p * 2 * ORC_D + ORC_D + d];
    double mu = orc_f16_to_double(cm[(p * ORC_NCHUNK + j) * 2 * ORC_D + d]);
    double s = orc_f16_to_double(cm[(p * ORC_NCHUNK + j) * 2 * ORC_D + ORC_D + d]);
    return mn + rng * (mu + s * sg * lvd[k]);
}

static void level_values(double *lvd)
{
    float thr[64];
    uint16_t lv[65];
    orc_tables(thr, lv);
    for (int k = 0; k <= 64; ++k)
        lvd[k] = orc_f16_to_double(lv[k]);
}

/* Dense reconstruction of a whole [L][H][T][128] tensor in fp64.
 * res == NULL (or full == 0) gives the anchor-only draft cache. */
int orc_dequant(const uint8_t *anc, const uint8_t *res, const float *pm, const uint16_t *cm, int L,
                int H, int T, int full, double *out)
{
    if (T % ORC_PAGE || (full && !res))
        return 1;
    double lvd[65];
    level_values(lvd);
    const int P = T / ORC_PAGE;
    const int64_t lhs = (int64_t)L * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t lh = 0; lh < lhs; ++lh) {
        const uint8_t *a = anc + (size_t)lh * T * (ORC_D / 2);
        const uint8_t *r = res ? res + (size_t)lh * T * (ORC_D / 2) : NULL;
        const float *p = pm + (size_t)lh * P * 2 * ORC_D;
        const uint16_t *c = cm + (size_t)lh * P * ORC_NCHUNK * 2 * ORC_D;
        double *o = out + (size_t)lh * T * ORC_D;
        for (size_t row = 0; row < (size_t)T; ++row)
            for (int d = 0; d < ORC_D; ++d)
                o[row * ORC_D + d] = decode_one(a, r, p, c, lvd, row, d, full);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* decode attention over the quantized paged cache, fp64               */
/* ------------------------------------------------------------------ */

/* One decode step for every request b and query head h of one layer.
 * q: [B][Hq][128] bf16 bits. K and V: planes and metadata of the whole
 * [L][H][T] pool; `layer` selects the layer. page_table: [B][max_pages]
 * physical page numbers (a page p is rows 256p..256p+255 of the pool).
 * ctx: [B] context lengths. Query head h reads KV head h / (Hq / H).
 * out: [B][Hq][128]; scores (optional): [B][Hq][max_pages*256] scaled logits
 * for t < ctx, -inf after. Returns 1 on a bad page number or length. */
int orc_decode_attn(const uint16_t *q, int B, int Hq, const uint8_t *ka, const uint8_t *kr,
                    const float *kpm, const uint16_t *kcm, const uint8_t *va, const uint8_t *vr,
                    const float *vpm, const uint16_t *vcm, int L, int H, int T, int layer,
                    const int32_t *page_table, const int32_t *ctx, int max_pages, double sm_scale,
                    int full, double *out, double *scores)
{
    if (H <= 0 || Hq % H || T % ORC_PAGE || layer < 0 || layer >= L)
        return 1;
    if (full && (!kr || !vr))
        return 1;
    const int G = Hq / H;
    const int P = T / ORC_PAGE;
    double lvd[65];
    level_values(lvd);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        if (ctx[b] < 0 || ctx[b] > max_pages * ORC_PAGE)
            bad = 1;
        for (int i = 0; ctx[b] > 0 && i < (ctx[b] + ORC_PAGE - 1) / ORC_PAGE && i < max_pages; ++i)
            if (page_table[(size_t)b * max_pages + i] < 0 || page_table[(size_t)b * max_pages + i] >= P)
                bad = 1;
    }
    if (bad)
        return 1;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < H; ++g) {
            const int n = ctx[b];
            const size_t lh = (size_t)layer * H + g;
            const uint8_t *a_k = ka + lh * T * (ORC_D / 2), *a_v = va + lh * T * (ORC_D / 2);
            const uint8_t *r_k = kr ? kr + lh * T * (ORC_D / 2) : NULL;
            const uint8_t *r_v = vr ? vr + lh * T * (ORC_D / 2) : NULL;
            const float *pk = kpm + lh * P * 2 * ORC_D, *pv = vpm + lh * P * 2 * ORC_D;
            const uint16_t *ck = kcm + lh * P * ORC_NCHUNK * 2 * ORC_D;
            const uint16_t *cv = vcm + lh * P * ORC_NCHUNK * 2 * ORC_D;
            double *s = n > 0 ? malloc(sizeof(double) * (size_t)n * G) : NULL;
            double kk[ORC_D], qd[ORC_D];
            for (int t = 0; t < n; ++t) {
                size_t row = (size_t)page_table[(size_t)b * max_pages + t / ORC_PAGE] * ORC_PAGE + t % ORC_PAGE;
                for (int d = 0; d < ORC_D; ++d)
                    kk[d] = decode_one(a_k, r_k, pk, ck, lvd, row, d, full);
                for (int h = 0; h < G; ++h) {
                    const uint16_t *qh = q + ((size_t)b * Hq + (size_t)g * G + h) * ORC_D;
                    double acc = 0.0;
                    for (int d = 0; d < ORC_D; ++d)
                        acc += (double)bf16_to_f32(qh[d]) * kk[d];
                    s[(size_t)t * G + h] = sm_scale * acc;
                }
            }
            for (int h = 0; h < G; ++h) {
                size_t hq = (size_t)b * Hq + (size_t)g * G + h;
                double *o = out + hq * ORC_D;
                for (int d = 0; d < ORC_D; ++d)
                    o[d] = 0.0;
                if (scores) {
                    double *sc = scores + hq * (size_t)max_pages * ORC_PAGE;
                    for (int t = 0; t < max_pages * ORC_PAGE; ++t)
                        sc[t] = t < n ? s[(size_t)t * G + h] : -INFINITY;
                }
                if (n == 0)
                    continue;
                double m = -INFINITY;
                for (int t = 0; t < n; ++t)
                    if (s[(size_t)t * G + h] > m)
                        m = s[(size_t)t * G + h];
                double l = 0.0;
                for (int t = 0; t < n; ++t) {
                    double p = exp(s[(size_t)t * G + h] - m);
                    s[(size_t)t * G + h] = p;
                    l += p;
                }
                for (int t = 0; t < n; ++t)
                    s[(size_t)t * G + h] /= l;
            }
            for (int t = 0; t < n; ++t) {
                size_t row = (size_t)page_table[(size_t)b * max_pages + t / ORC_PAGE] * ORC_PAGE + t % ORC_PAGE;
                for (int d = 0; d < ORC_D; ++d)
                    kk[d] = decode_one(a_v, r_v, pv, cv, lvd, row, d, full);
                for (int h = 0; h < G; ++h) {
                    double p = s[(size_t)t * G + h];
                    double *o = out + ((size_t)b * Hq + (size_t)g * G + h) * ORC_D;
                    for (int d = 0; d < ORC_D; ++d)
                        o[d] += p * kk[d];
                }
            }
            (void)qd;
            free(s);
        }
    }
    return 0;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
