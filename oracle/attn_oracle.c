/*
 * attn_oracle.c -- plain fp64 CPU attention forward.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the correctness oracle for the bf16 attention forward library in this
 * repository.  Only the test suite, the package's smoke check and the CPU-baseline leg of
 * the benchmark load it; the product path never does.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Source pages (cited by short name):
 *   [MoonMath]  "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats
 *               AITER" (news.chathome.org).
 *               - opening section: attention is the fused softmax(Q K^T / sqrt(d)) V;
 *                 bf16 forward, BSHD or BHSD, no transposes, head dim 128, arbitrary
 *                 sequence lengths including cross-attention;
 *               - opening section, limitations paragraph: three output rounding modes
 *                 (RTNE, RTNA, RTZ), NaN/Inf handling bitwise identical, deterministic.
 *
 * What is computed, per output row (b, h, i), with no blocking, fusion or online rescaling:
 *   s_j   = (sum_x q_x k_{j,x}) * (1/sqrt(d))               x = 0..d-1 in order, fp64
 *   rows with a NaN or +inf logit, or with every logit -inf, are all NaN;
 *   m     = max of the finite s_j
 *   w_j   = exp(s_j - m) for finite s_j, 0 for s_j = -inf
 *   l     = sum_j w_j
 *   O_x   = (sum_j w_j v_{j,x}) / l
 * with exact-arithmetic treatment of non-finite V: a key with a finite logit has a strictly
 * positive weight even when exp() underflows in fp64 (so w * inf = inf), and a key with a
 * -inf logit contributes 0 * v (NaN when v is not finite).  The result is rounded once,
 * from fp64 straight to bf16, in the requested mode; every NaN becomes 0x7FC0.
 *
 * The readings above (IEEE meaning of the formula for non-finite inputs, the three mode
 * names as IEEE roundTiesToEven / roundTiesToAway / roundTowardZero on the final value)
 * are where the pages are silent; they are listed with the other readings in the design
 * notes of this repository.
 *
 * Extensions named by the same article's limitations paragraph (causal masking and GQA are
 * listed there as not yet supported by the MI300X kernel):
 *   - causal: key j is visible to query i iff j <= i + (Skv - Sq) (aligned at the last
 *     query/key; plain causal when Sq = Skv).  Masked keys are left out of the row entirely;
 *     a row with no visible key is NaN (empty softmax) with log-sum-exp -inf.
 *   - grouped K/V heads: Hkv divides H, and query head h reads K/V head h / (H / Hkv).
 *   - lse: natural log of sum_j exp(s_j) over the visible keys; NaN for a row holding a NaN
 *     or +inf logit, -inf when every visible logit is -inf or no key is visible.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_LAYOUT_BSHD 0
#define ORACLE_LAYOUT_BHSD 1
#define ORACLE_ROUND_RTNE 0
#define ORACLE_ROUND_RTNA 1
#define ORACLE_ROUND_RTZ 2

/* bf16 bit pattern -> exact double.  A bf16 value is the top half of an fp32 value. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Offset (in elements) of element (b, s, h, x) for the given layout.
 * BSHD: ((b*S + s)*H + h)*d + x      BHSD: ((b*H + h)*S + s)*d + x
 * [MoonMath] opening section: the kernel reads BSHD or BHSD tensors as they are. */
static int64_t elem_offset(int layout, int64_t b, int64_t s, int64_t h, int64_t x,
                           int64_t S, int64_t H, int64_t d) {
    if (layout == ORACLE_LAYOUT_BSHD) return ((b * S + s) * H + h) * d + x;
    return ((b * H + h) * S + s) * d + x;
}

/*
 * Round a double to the nearest bf16 in the given mode, returning the bit pattern.
 * [MoonMath] limitations paragraph: output rounding in RTNE, RTNA or RTZ.
 * The quantum of the binade containing |x| is q = 2^(max(e,-126) - 7) where
 * e = floor(log2 |x|); a = |x| truncated to a multiple of q, b = a + q.  All of these are
 * exact in fp64 for every finite double.  Every NaN maps to the canonical 0x7FC0.
 */
uint16_t oracle_round_bf16(double x, int mode) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7F80;
    if (ax == 0.0) return sign;
    int fe;
    (void)frexp(ax, &fe);           /* ax = f * 2^fe, f in [0.5, 1) */
    int e = fe - 1;                 /* floor(log2 ax) */
    if (e > 127) {                  /* beyond every finite bf16 */
        return (uint16_t)(sign | (mode == ORACLE_ROUND_RTZ ? 0x7F7F : 0x7F80));
    }
    int qe = (e < -126 ? -126 : e) - 7;
    double q = ldexp(1.0, qe);
    double n = floor(ldexp(ax, -qe));   /* integer significand of the truncation */
    double a = ldexp(n, qe);
    double rem = ax - a;                /* exact: 0 <= rem < q */
    double half = 0.5 * q;
    double r = a;
    if (mode == ORACLE_ROUND_RTNE) {
        if (rem > half || (rem == half && fmod(n, 2.0) != 0.0)) r = a + q;
    } else if (mode == ORACLE_ROUND_RTNA) {
        if (rem >= half) r = a + q;
    } /* RTZ: r = a */
    /* r is now a bf16 value or 2^128 (overflow). */
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float rf = (float)r;                /* exact: every bf16 value is an fp32 value */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* Per-row work.  Outputs for the row are written at slot `slot` (row-major, d wide). */
static void oracle_row(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       int64_t b, int64_t h, int64_t i,
                       int64_t H, int64_t Hkv, int64_t Sq, int64_t Skv, int64_t d, int causal,
                       int layout, int mode,
                       double* s, double* w, double* qrow,
                       uint16_t* o_bits, double* o_f64, double* a_bound, double* lse,
                       double* probs, int64_t slot) {
    const double scale = 1.0 / sqrt((double)d);
    for (int64_t x = 0; x < d; ++x)
        qrow[x] = bf16_bits_to_double(q[elem_offset(layout, b, i, h, x, Sq, H, d)]);

    /* Visible keys: all, or with the causal mask keys 0 .. i + (Skv - Sq). */
    int64_t nvis = Skv;
    if (causal) {
        const int64_t last = i + (Skv - Sq);
        nvis = last < 0 ? 0 : (last + 1 < Skv ? last + 1 : Skv);
    }
    const int64_t kvh = h / (H / Hkv);   /* grouped K/V head read by query head h */

    /* Logits, [MoonMath] opening section: Q K^T / sqrt(d). */
    int any_nan_or_posinf = 0, all_neginf = 1;
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        double acc = 0.0;
        const int64_t kb = elem_offset(layout, b, j, kvh, 0, Skv, Hkv, d);
        for (int64_t x = 0; x < d; ++x) acc += qrow[x] * bf16_bits_to_double(k[kb + x]);
        s[j] = acc * scale;
        if (isnan(s[j]) || (isinf(s[j]) && s[j] > 0)) any_nan_or_posinf = 1;
        if (!(isinf(s[j]) && s[j] < 0)) all_neginf = 0;
        if (isfinite(s[j]) && s[j] > m) m = s[j];
    }

    if (any_nan_or_posinf || all_neginf) {
        /* softmax of a row holding NaN or +inf, or only -inf (or no visible key), is NaN
         * everywhere; its log-sum-exp is NaN, or -inf (log 0) when nothing but -inf is seen */
        for (int64_t x = 0; x < d; ++x) {
            o_bits[slot * d + x] = 0x7FC0;
            if (o_f64) o_f64[slot * d + x] = NAN;
            if (a_bound) a_bound[slot * d + x] = NAN;
        }
        if (lse) lse[slot] = any_nan_or_posinf ? NAN : -INFINITY;
        if (probs)
            for (int64_t j = 0; j < Skv; ++j) probs[slot * Skv + j] = NAN;
        return;
    }

    /* Weights relative to the row maximum: exp(s_j - m), 0 for -inf logits. */
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        w[j] = isfinite(s[j]) ? exp(s[j] - m) : 0.0;
        l += w[j];
    }
    if (lse) lse[slot] = m + log(l);
    if (probs)
        for (int64_t j = 0; j < Skv; ++j) probs[slot * Skv + j] = j < nvis ? w[j] / l : 0.0;

    for (int64_t x = 0; x < d; ++x) {
        double num = 0.0, absnum = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double vj = bf16_bits_to_double(v[elem_offset(layout, b, j, kvh, x, Skv, Hkv, d)]);
            double term;
            if (!isfinite(s[j])) {
                term = 0.0 * vj;                 /* -inf logit: weight exactly 0 */
            } else if (isinf(vj)) {
                term = vj;                       /* positive weight times +-inf */
            } else {
                term = w[j] * vj;                /* NaN in v propagates */
                absnum += w[j] * fabs(vj);
            }
            num += term;
        }
        const double ox = num / l;
        o_bits[slot * d + x] = oracle_round_bf16(ox, mode);
        if (o_f64) o_f64[slot * d + x] = ox;
        if (a_bound) a_bound[slot * d + x] = isfinite(ox) ? absnum / l : NAN;
    }
}

/*
 * attn_oracle_ex -- reference attention forward in fp64.
 *
 * q, k, v   bf16 bit patterns in `layout` (0 = BSHD, 1 = BHSD); q has Sq rows per (b, h)
 *           over H heads, k and v have Skv rows per (b, kv head) over Hkv heads (Hkv | H).
 * causal    0: every key visible; 1: key j visible to query i iff j <= i + (Skv - Sq).
 * rows      optional list of nrows flat row indices r = (b*H + h)*Sq + i; NULL means every
 *           row, in that (b, h, i) order.
 * o_bits    out, [nrows][d] bf16 bit patterns in list order.
 * o_f64     optional out, [nrows][d] unrounded result.
 * a_bound   optional out, [nrows][d] A = sum_j w_j |v_jx| / l (forward-error scale).
 * lse       optional out, [nrows] natural-log log-sum-exp of the visible scaled logits.
 * probs     optional out, [nrows][Skv] softmax weights w_j / l.
 * nthreads  OpenMP threads (<= 0: runtime default).
 * Returns 0 on success, -1 on bad arguments.
 */
int attn_oracle_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   int64_t B, int64_t H, int64_t Hkv, int64_t Sq, int64_t Skv, int64_t d,
                   int layout, int mode, int causal, const int64_t* rows, int64_t nrows,
                   uint16_t* o_bits, double* o_f64, double* a_bound, double* lse,
                   double* probs, int nthreads) {
    if (!q || !k || !v || !o_bits) return -1;
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 1 || Skv < 1 || d < 1) return -1;
    if (causal != 0 && causal != 1) return -1;
    if (layout != ORACLE_LAYOUT_BSHD && layout != ORACLE_LAYOUT_BHSD) return -1;
    if (mode < ORACLE_ROUND_RTNE || mode > ORACLE_ROUND_RTZ) return -1;
    const int64_t total = B * H * Sq;
    const int64_t n = rows ? nrows : total;
    if (rows)
        for (int64_t r = 0; r < n; ++r)
            if (rows[r] < 0 || rows[r] >= total) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Skv);
        double* w = (double*)malloc(sizeof(double) * (size_t)Skv);
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !w || !qrow) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n; ++r) {
                const int64_t flat = rows ? rows[r] : r;
                const int64_t i = flat % Sq;
                const int64_t h = (flat / Sq) % H;
                const int64_t b = flat / (Sq * H);
                oracle_row(q, k, v, b, h, i, H, Hkv, Sq, Skv, d, causal, layout, mode, s, w,
                           qrow, o_bits, o_f64, a_bound, lse, probs, r);
            }
        }
        free(s);
        free(w);
        free(qrow);
    }
    return bad ? -1 : 0;
}

/* attn_oracle_ex with one K/V head per query head and no mask. */
int attn_oracle(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t d,
                int layout, int mode, const int64_t* rows, int64_t nrows,
                uint16_t* o_bits, double* o_f64, double* a_bound, double* lse,
                double* probs, int nthreads) {
    return attn_oracle_ex(q, k, v, B, H, H, Sq, Skv, d, layout, mode, 0, rows, nrows, o_bits,
                          o_f64, a_bound, lse, probs, nthreads);
}

/* Batch rounding helper so the rounding rule can be tested on its own. */
void oracle_round_bf16_array(const double* x, int64_t n, int mode, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i], mode);
}

/* Threads OpenMP would use by default (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
