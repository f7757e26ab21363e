/*
 * attn_oracle_bwd.c -- plain fp64 CPU attention backward, and a forward on fp64 inputs.
 * TEST INFRASTRUCTURE ONLY (the same rules as attn_oracle.c: only the test suite, the smoke
 * check and the benchmark's CPU leg load it; it shares no code with the CUDA path).
 *
 * Source pages (cited by short name):
 *   [HipKittens] "HipKittens: Fast and Furious AMD Kernels (MLSys 2026)", "Key observations"
 *               (observation 3) and "Attention backward": the attention backward -- the
 *               gradients of softmax(Q K^T / sqrt(d)) V with respect to Q, K and V -- is the
 *               next kernel after the forward.
 *   [MoonMath]  "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats
 *               AITER", opening section: the forward being differentiated.
 *
 * What is computed.  With c = 1/sqrt(d), for every query row i of a (b, h) and its visible
 * keys j (all keys, or j <= i + Skv - Sq with the causal mask), in fp64:
 *   s_ij = c q_i . k_j,   p_ij = exp(s_ij - m_i) / sum_j exp(s_ij - m_i),   O_i = sum_j p_ij v_j
 * and, for an upstream gradient dO (the derivative of a scalar loss with respect to O):
 *   dV_j  = sum_i p_ij dO_i                      (over the rows, and the query heads, that
 *                                                 see key j of K/V head kvh)
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_x dO_ix O_ix                     (= sum_j p_ij dP_ij)
 *   dS_ij = p_ij (dP_ij - D_i)                   (the softmax Jacobian applied to dP)
 *   dQ_i  = c sum_j dS_ij k_j
 *   dK_j  = c sum_i dS_ij q_i
 * These are the chain rule through O = P V, P = softmax(S) and S = c Q K^T, written out;
 * the pins check them against numerical differentiation of attn_oracle_f64_forward.
 * A query with no visible key contributes nothing (its dQ row is 0).  Inputs are expected
 * finite; IEEE arithmetic propagates anything else.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define BWD_LAYOUT_BSHD 0

static double bwd_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Offset of element (b, s, h, x): BSHD ((b*S + s)*H + h)*d + x, BHSD ((b*H + h)*S + s)*d + x */
static int64_t bwd_offset(int layout, int64_t b, int64_t s, int64_t h, int64_t x,
                          int64_t S, int64_t H, int64_t d) {
    if (layout == BWD_LAYOUT_BSHD) return ((b * S + s) * H + h) * d + x;
    return ((b * H + h) * S + s) * d + x;
}

static int64_t visible_keys(int causal, int64_t i, int64_t Sq, int64_t Skv) {
    if (!causal) return Skv;
    const int64_t last = i + (Skv - Sq);
    return last < 0 ? 0 : (last + 1 < Skv ? last + 1 : Skv);
}

static int bad_shape(int64_t B, int64_t H, int64_t Hkv, int64_t Sq, int64_t Skv, int64_t d,
                     int layout, int causal) {
    return B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Sq < 1 || Skv < 1 || d < 1 ||
           (layout != 0 && layout != 1) || (causal != 0 && causal != 1);
}

/*
 * attn_oracle_f64_forward -- O = softmax(c Q K^T) V on fp64 inputs (no rounding), the
 * function whose derivative the backward is.  q, k, v, o in `layout`; returns 0, or -1 on
 * bad arguments.  Rows with no visible key are 0 here (they carry no dependence).
 */
int attn_oracle_f64_forward(const double* q, const double* k, const double* v, int64_t B,
                            int64_t H, int64_t Hkv, int64_t Sq, int64_t Skv, int64_t d,
                            int layout, int causal, double* o) {
    if (!q || !k || !v || !o || bad_shape(B, H, Hkv, Sq, Skv, d, layout, causal)) return -1;
    const double c = 1.0 / sqrt((double)d);
    int bad = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Skv);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < B * H * Sq; ++r) {
                const int64_t b = r / (H * Sq), h = (r / Sq) % H, i = r % Sq;
                const int64_t kvh = h / (H / Hkv), nvis = visible_keys(causal, i, Sq, Skv);
                double m = -INFINITY;
                for (int64_t j = 0; j < nvis; ++j) {
                    double acc = 0.0;
                    for (int64_t x = 0; x < d; ++x)
                        acc += q[bwd_offset(layout, b, i, h, x, Sq, H, d)] *
                               k[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)];
                    s[j] = c * acc;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < nvis; ++j) {
                    s[j] = exp(s[j] - m);
                    l += s[j];
                }
                for (int64_t x = 0; x < d; ++x) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < nvis; ++j)
                        acc += s[j] * v[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)];
                    o[bwd_offset(layout, b, i, h, x, Sq, H, d)] = nvis ? acc / l : 0.0;
                }
            }
            free(s);
        }
    }
    return bad ? -1 : 0;
}

/*
 * attn_oracle_bwd -- the gradients above for bf16 inputs q, k, v and upstream gradient
 * dout (bf16, laid out like q), all in `layout`.
 *   dq [like q], dk, dv [like k / v]     fp64 outputs (required)
 *   dq_a, dk_a, dv_a                     optional fp64 forward-error scales, same shapes:
 *                                        dV: sum_i p_ij |dO_ix|
 *                                        dQ: c sum_j p_ij (|dP_ij| + |D|_i) |k_jx|
 *                                        dK: c sum_i p_ij (|dP_ij| + |D|_i) |q_ix|
 *                                        with |D|_i = sum_x |dO_ix| |O_ix| (the sums of the
 *                                        terms' magnitudes; dS is bounded by p (|dP| + |D|),
 *                                        and |D| also bounds D's error when it is formed from
 *                                        a rounded O)
 *   delta                                optional fp64 [B][H][Sq]: D_i
 * Work is split over (b, K/V head): each owns its dK and dV rows and the dQ rows of the
 * query heads that read it, so no two threads write the same output.
 * Returns 0, or -1 on bad arguments.
 */
int attn_oracle_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* dout, int64_t B, int64_t H, int64_t Hkv, int64_t Sq,
                    int64_t Skv, int64_t d, int layout, int causal, double* dq, double* dk,
                    double* dv, double* dq_a, double* dk_a, double* dv_a, double* delta,
                    int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if (bad_shape(B, H, Hkv, Sq, Skv, d, layout, causal)) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const double c = 1.0 / sqrt((double)d);
    const int64_t group = H / Hkv;
    memset(dk, 0, sizeof(double) * (size_t)(B * Hkv * Skv * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * Hkv * Skv * d));
    if (dk_a) memset(dk_a, 0, sizeof(double) * (size_t)(B * Hkv * Skv * d));
    if (dv_a) memset(dv_a, 0, sizeof(double) * (size_t)(B * Hkv * Skv * d));
    int bad = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)Skv);
        double* dp = (double*)malloc(sizeof(double) * (size_t)Skv);
        double* qi = (double*)malloc(sizeof(double) * (size_t)d);
        double* gi = (double*)malloc(sizeof(double) * (size_t)d);
        if (!p || !dp || !qi || !gi) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bk = 0; bk < B * Hkv; ++bk) {
                const int64_t b = bk / Hkv, kvh = bk % Hkv;
                for (int64_t h = kvh * group; h < (kvh + 1) * group; ++h) {
                    for (int64_t i = 0; i < Sq; ++i) {
                        const int64_t nvis = visible_keys(causal, i, Sq, Skv);
                        for (int64_t x = 0; x < d; ++x) {
                            qi[x] = bwd_bits_to_double(q[bwd_offset(layout, b, i, h, x, Sq, H, d)]);
                            gi[x] = bwd_bits_to_double(dout[bwd_offset(layout, b, i, h, x, Sq, H, d)]);
                        }
                        /* probabilities of the visible keys */
                        double m = -INFINITY;
                        for (int64_t j = 0; j < nvis; ++j) {
                            double acc = 0.0;
                            for (int64_t x = 0; x < d; ++x)
                                acc += qi[x] * bwd_bits_to_double(k[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)]);
                            p[j] = c * acc;
                            if (p[j] > m) m = p[j];
                        }
                        double l = 0.0;
                        for (int64_t j = 0; j < nvis; ++j) {
                            p[j] = exp(p[j] - m);
                            l += p[j];
                        }
                        for (int64_t j = 0; j < nvis; ++j) p[j] /= l;
                        /* dP_ij = dO_i . v_j and D_i = sum_j p_ij dP_ij (= dO_i . O_i) */
                        double Di = 0.0;
                        for (int64_t j = 0; j < nvis; ++j) {
                            double acc = 0.0;
                            for (int64_t x = 0; x < d; ++x)
                                acc += gi[x] * bwd_bits_to_double(v[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)]);
                            dp[j] = acc;
                            Di += p[j] * acc;
                        }
                        /* |D|_i = sum_x |dO_ix| |O_ix| for the error scales */
                        double Dabs = 0.0;
                        if (dq_a || dk_a)
                            for (int64_t x = 0; x < d; ++x) {
                                double ox = 0.0;
                                for (int64_t j = 0; j < nvis; ++j)
                                    ox += p[j] * bwd_bits_to_double(v[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)]);
                                Dabs += fabs(gi[x]) * fabs(ox);
                            }
                        if (delta) delta[(b * H + h) * Sq + i] = Di;
                        /* dQ_i = c sum_j p_ij (dP_ij - D_i) k_j */
                        for (int64_t x = 0; x < d; ++x) {
                            double acc = 0.0, mag = 0.0;
                            for (int64_t j = 0; j < nvis; ++j) {
                                const double kjx = bwd_bits_to_double(k[bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d)]);
                                acc += p[j] * (dp[j] - Di) * kjx;
                                mag += p[j] * (fabs(dp[j]) + Dabs) * fabs(kjx);
                            }
                            const int64_t off = bwd_offset(layout, b, i, h, x, Sq, H, d);
                            dq[off] = c * acc;
                            if (dq_a) dq_a[off] = c * mag;
                        }
                        /* dK_j += c dS_ij q_i,  dV_j += p_ij dO_i */
                        for (int64_t j = 0; j < nvis; ++j) {
                            const double ds = p[j] * (dp[j] - Di);
                            const double dsa = p[j] * (fabs(dp[j]) + Dabs);
                            for (int64_t x = 0; x < d; ++x) {
                                const int64_t off = bwd_offset(layout, b, j, kvh, x, Skv, Hkv, d);
                                dk[off] += c * ds * qi[x];
                                dv[off] += p[j] * gi[x];
                                if (dk_a) dk_a[off] += c * dsa * fabs(qi[x]);
                                if (dv_a) dv_a[off] += p[j] * fabs(gi[x]);
                            }
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
        free(qi);
        free(gi);
    }
    return bad ? -1 : 0;
}
