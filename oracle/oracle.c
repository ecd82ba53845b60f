/*
 * fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition, with no tiling, no online softmax
 * and no reordering beyond what the definition states:
 *
 *   "FlashAttention Primer" (oripoin.me), section "Why attention is quadratic",
 *   the SDPA equation:      S = Q K^T * scale,  P = rowsoftmax(S),  O = P V
 *   "Flash Attention" (aiwiki.ai), section "Definition and scope": the same map.
 *
 * The saved per-row statistic is the natural-log log-sum-exp of the scaled
 * scores, LSE_i = m_i + ln(l_i) ("FlashAttention Primer", section "Backward pass:
 * recomputation instead of storage", which saves O and a per-row log-sum-exp).
 *
 * Backward: the gradient of O = softmax(scale Q K^T) V with upstream dO.
 *   dV_k = sum_i P_ik dO_i
 *   dP_ik = dO_i . v_k
 *   D_i  = sum_c dO_ic O_ic  (= sum_k P_ik dP_ik)
 *   dS_ik = P_ik (dP_ik - D_i)
 *   dQ_i = scale sum_k dS_ik k_k,   dK_k = scale sum_i dS_ik q_i
 * The primer's printed backward (Figure 5 and the equation above it) drops the
 * -D_i term of the softmax Jacobian and the scale factor; this oracle keeps both
 * (the gradient of the definition), and the tests pin it against finite
 * differences of the forward, which does not depend on this formula.
 *
 * Grouped-query attention: query head h reads KV head floor(h * Hkv / Hq)
 * (contiguous groups, "Flash Attention" (aiwiki.ai), section "FlashAttention-2",
 * which covers MQA/GQA where several query heads share one KV head).  dK and dV
 * of a KV head are the sums over its query heads.
 *
 * Causal: key k is visible to query i iff k <= i ("FlashAttention Primer",
 * section "FlashAttention-1", causal masking paragraph: future scores are -inf).
 *
 * Layouts (all row-major, fp64):
 *   q, o, dO, dq : [B, Hq, N, d]      k, v, dk, dv : [B, Hkv, N, d]
 *   lse, D       : [B, Hq, N]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static int check_args(int B, int Hq, int Hkv, int N, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0) return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int oracle_num_threads_in_team(void) {
#ifdef _OPENMP
    return omp_get_num_threads();
#else
    return 1;
#endif
}

static double dot(const double* a, const double* b, int d) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/*
 * One query row of one head: fills p[0..nk) with the normalised softmax row over
 * the nk visible keys and returns the row's log-sum-exp.  Plain max-shifted
 * softmax, evaluated in fp64.
 */
static double softmax_row(const double* qi, const double* kh, int nk, int d,
                          double scale, double* p) {
    double m = -INFINITY;
    for (int k = 0; k < nk; ++k) {
        p[k] = scale * dot(qi, kh + (size_t)k * d, d);
        if (p[k] > m) m = p[k];
    }
    double l = 0.0;
    for (int k = 0; k < nk; ++k) {
        p[k] = exp(p[k] - m);
        l += p[k];
    }
    for (int k = 0; k < nk; ++k) p[k] /= l;
    return m + log(l);
}

int oracle_forward(const double* q, const double* k, const double* v, double* o,
                   double* lse, int B, int Hq, int Hkv, int N, int d, int causal,
                   double scale) {
    int rc = check_args(B, Hq, Hkv, N, d);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    const int64_t rows = (int64_t)B * Hq * N;
    int failed = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!p) continue;
            const int i = (int)(r % N);
            const int64_t bh = r / N;
            const int h = (int)(bh % Hq);
            const int b = (int)(bh / Hq);
            const int g = (int)(((int64_t)h * Hkv) / Hq);
            const double* qi = q + (size_t)r * d;
            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;
            const double* vh = v + ((size_t)b * Hkv + g) * (size_t)N * d;
            const int nk = causal ? i + 1 : N;
            lse[r] = softmax_row(qi, kh, nk, d, scale, p);
            double* oi = o + (size_t)r * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int kk = 0; kk < nk; ++kk) {
                const double w = p[kk];
                const double* vk = vh + (size_t)kk * d;
                for (int c = 0; c < d; ++c) oi[c] += w * vk[c];
            }
        }
        free(p);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * Sliding-window (local) causal attention: key k is visible to query i iff
 * i - window < k <= i ("Flash Attention" (aiwiki.ai), section "Features":
 * local sliding windows; block-sparse attention skips the blocks a mask
 * leaves empty, section "Block-sparse FlashAttention").  window >= N is
 * ordinary causal attention.  Layouts as for oracle_forward / oracle_backward.
 */
static double softmax_row_from(const double* qi, const double* kh, int k0, int k1, int d,
                               double scale, double* p) {
    /* p[0 .. k1-k0) over keys k0 .. k1-1 */
    return softmax_row(qi, kh + (size_t)k0 * d, k1 - k0, d, scale, p);
}

int oracle_forward_window(const double* q, const double* k, const double* v, double* o,
                          double* lse, int B, int Hq, int Hkv, int N, int d, int window,
                          double scale) {
    int rc = check_args(B, Hq, Hkv, N, d);
    if (rc) return rc;
    if (window < 1 || !q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    const int64_t rows = (int64_t)B * Hq * N;
    int failed = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!p) continue;
            const int i = (int)(r % N);
            const int64_t bh = r / N;
            const int h = (int)(bh % Hq);
            const int b = (int)(bh / Hq);
            const int g = (int)(((int64_t)h * Hkv) / Hq);
            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;
            const double* vh = v + ((size_t)b * Hkv + g) * (size_t)N * d;
            const int k0 = i - window + 1 > 0 ? i - window + 1 : 0;
            lse[r] = softmax_row_from(q + (size_t)r * d, kh, k0, i + 1, d, scale, p);
            double* oi = o + (size_t)r * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int kk = k0; kk <= i; ++kk)
                for (int c = 0; c < d; ++c) oi[c] += p[kk - k0] * vh[(size_t)kk * d + c];
        }
        free(p);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

int oracle_backward_window(const double* q, const double* k, const double* v, const double* dO,
                           double* dq, double* dk, double* dv, int B, int Hq, int Hkv, int N,
                           int d, int window, double scale) {
    int rc = check_args(B, Hq, Hkv, N, d);
    if (rc) return rc;
    if (window < 1 || !q || !k || !v || !dO || !dq || !dk || !dv) return ORACLE_EINVAL;
    const int group = Hq / Hkv;
    const size_t nd = (size_t)N * d;
    /* One KV head at a time, its group's rows in order (small sizes only). */
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    double* ds = (double*)malloc(sizeof(double) * (size_t)N);
    double* oi = (double*)malloc(sizeof(double) * (size_t)d);
    if (!p || !ds || !oi) {
        free(p);
        free(ds);
        free(oi);
        return ORACLE_ENOMEM;
    }
    for (int64_t bg = 0; bg < (int64_t)B * Hkv; ++bg) {
        const int64_t b = bg / Hkv;
        const int g = (int)(bg % Hkv);
        const double* kh = k + (size_t)bg * nd;
        const double* vh = v + (size_t)bg * nd;
        double* dkh = dk + (size_t)bg * nd;
        double* dvh = dv + (size_t)bg * nd;
        memset(dkh, 0, sizeof(double) * nd);
        memset(dvh, 0, sizeof(double) * nd);
        for (int hh = 0; hh < group; ++hh) {
            const int h = g * group + hh;
            for (int i = 0; i < N; ++i) {
                const size_t row = ((size_t)b * Hq + h) * (size_t)N + i;
                const double* qi = q + row * d;
                const double* doi = dO + row * d;
                double* dqi = dq + row * d;
                const int k0 = i - window + 1 > 0 ? i - window + 1 : 0;
                const int nk = i + 1 - k0;
                softmax_row_from(qi, kh, k0, i + 1, d, scale, p);
                for (int c = 0; c < d; ++c) oi[c] = 0.0;
                for (int t = 0; t < nk; ++t)
                    for (int c = 0; c < d; ++c) oi[c] += p[t] * vh[(size_t)(k0 + t) * d + c];
                const double Di = dot(doi, oi, d);
                for (int t = 0; t < nk; ++t) ds[t] = p[t] * (dot(doi, vh + (size_t)(k0 + t) * d, d) - Di);
                for (int c = 0; c < d; ++c) dqi[c] = 0.0;
                for (int t = 0; t < nk; ++t)
                    for (int c = 0; c < d; ++c) dqi[c] += ds[t] * kh[(size_t)(k0 + t) * d + c];
                for (int c = 0; c < d; ++c) dqi[c] *= scale;
                for (int t = 0; t < nk; ++t) {
                    double* dkk = dkh + (size_t)(k0 + t) * d;
                    double* dvk = dvh + (size_t)(k0 + t) * d;
                    for (int c = 0; c < d; ++c) {
                        dkk[c] += scale * ds[t] * qi[c];
                        dvk[c] += p[t] * doi[c];
                    }
                }
            }
        }
    }
    free(p);
    free(ds);
    free(oi);
    return ORACLE_OK;
}

/*
 * Forward with Nq query rows and Nk keys per head (non-causal): the same
 * definition with a rectangular score matrix, as used for decoding, where a
 * few new query rows attend to a long sequence of cached keys.
 *   q, o : [B, Hq, Nq, d]    k, v : [B, Hkv, Nk, d]    lse : [B, Hq, Nq]
 */
int oracle_forward_rect(const double* q, const double* k, const double* v, double* o,
                        double* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        double scale) {
    int rc = check_args(B, Hq, Hkv, Nq, d);
    if (rc) return rc;
    if (Nk <= 0) return ORACLE_EINVAL;
    if (!q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    const int64_t rows = (int64_t)B * Hq * Nq;
    int failed = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)Nk);
        if (!p) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < rows; ++r) {
            if (!p) continue;
            const int64_t bh = r / Nq;
            const int h = (int)(bh % Hq);
            const int b = (int)(bh / Hq);
            const int g = (int)(((int64_t)h * Hkv) / Hq);
            const double* qi = q + (size_t)r * d;
            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            const double* vh = v + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            lse[r] = softmax_row(qi, kh, Nk, d, scale, p);
            double* oi = o + (size_t)r * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int kk = 0; kk < Nk; ++kk)
                for (int c = 0; c < d; ++c) oi[c] += p[kk] * vh[(size_t)kk * d + c];
        }
        free(p);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * Backward from the definition.  Recomputes P and O itself from (q, k, v); it
 * takes no forward output from anywhere else.  D (may be NULL) receives
 * D_i = dO_i . O_i.  KV heads are processed one after another; within one, the
 * rows of its query-head group are spread over threads, each summing its rows'
 * dK / dV contributions into a private buffer, and the buffers are added in
 * thread order at the end (the definition's sums over rows are order-free).
 */
int oracle_backward(const double* q, const double* k, const double* v, const double* dO,
                    double* dq, double* dk, double* dv, double* D, int B, int Hq,
                    int Hkv, int N, int d, int causal, double scale) {
    int rc = check_args(B, Hq, Hkv, N, d);
    if (rc) return rc;
    if (!q || !k || !v || !dO || !dq || !dk || !dv) return ORACLE_EINVAL;
    const int group = Hq / Hkv;
    const int64_t heads = (int64_t)B * Hkv;
    const size_t nd = (size_t)N * d;
    int failed = 0;
    for (int64_t bg = 0; bg < heads && !failed; ++bg) {
        const int64_t b = bg / Hkv;
        const int g = (int)(bg % Hkv);
        const double* kh = k + (size_t)bg * nd;
        const double* vh = v + (size_t)bg * nd;
        double* dkh = dk + (size_t)bg * nd;
        double* dvh = dv + (size_t)bg * nd;
        memset(dkh, 0, sizeof(double) * nd);
        memset(dvh, 0, sizeof(double) * nd);
        const int64_t rows = (int64_t)group * N;
#pragma omp parallel
        {
            double* p = (double*)malloc(sizeof(double) * (size_t)N);
            double* ds = (double*)malloc(sizeof(double) * (size_t)N);
            double* oi = (double*)malloc(sizeof(double) * (size_t)d);
            double* dk_part = (double*)calloc(nd, sizeof(double));
            double* dv_part = (double*)calloc(nd, sizeof(double));
            const int ok = p && ds && oi && dk_part && dv_part;
            if (!ok) {
#pragma omp atomic write
                failed = 1;
            }
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < rows; ++r) {
                if (!ok) continue;
                const int hh = (int)(r / N);
                const int i = (int)(r % N);
                const int h = g * group + hh;
                const size_t row = ((size_t)b * Hq + h) * (size_t)N + i;
                const double* qi = q + row * d;
                const double* doi = dO + row * d;
                double* dqi = dq + row * d;
                const int nk = causal ? i + 1 : N;
                softmax_row(qi, kh, nk, d, scale, p);
                /* O_i = sum_k P_ik v_k, then D_i = dO_i . O_i */
                for (int c = 0; c < d; ++c) oi[c] = 0.0;
                for (int kk = 0; kk < nk; ++kk)
                    for (int c = 0; c < d; ++c) oi[c] += p[kk] * vh[(size_t)kk * d + c];
                const double Di = dot(doi, oi, d);
                if (D) D[row] = Di;
                /* dS_ik = P_ik (dO_i . v_k - D_i) */
                for (int kk = 0; kk < nk; ++kk)
                    ds[kk] = p[kk] * (dot(doi, vh + (size_t)kk * d, d) - Di);
                /* dQ_i = scale sum_k dS_ik k_k */
                for (int c = 0; c < d; ++c) dqi[c] = 0.0;
                for (int kk = 0; kk < nk; ++kk)
                    for (int c = 0; c < d; ++c) dqi[c] += ds[kk] * kh[(size_t)kk * d + c];
                for (int c = 0; c < d; ++c) dqi[c] *= scale;
                /* dK_k += scale dS_ik q_i ; dV_k += P_ik dO_i */
                for (int kk = 0; kk < nk; ++kk) {
                    const double a = scale * ds[kk];
                    const double w = p[kk];
                    double* dkk = dk_part + (size_t)kk * d;
                    double* dvk = dv_part + (size_t)kk * d;
                    for (int c = 0; c < d; ++c) {
                        dkk[c] += a * qi[c];
                        dvk[c] += w * doi[c];
                    }
                }
            }
#pragma omp for ordered schedule(static, 1)
            for (int tt = 0; tt < oracle_num_threads_in_team(); ++tt) {
#pragma omp ordered
                if (ok) {
                    for (size_t e = 0; e < nd; ++e) {
                        dkh[e] += dk_part[e];
                        dvh[e] += dv_part[e];
                    }
                }
            }
            free(p);
            free(ds);
            free(oi);
            free(dk_part);
            free(dv_part);
        }
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* ==================================================================== FP8 (e4m3) inputs
 *
 * The low-precision forward of FlashAttention-3 ("FlashAttention Primer", section
 * "FlashAttention-3: Hopper asynchrony and FP8": block quantization and an incoherent
 * rotation applied before quantization; "Flash Attention" (aiwiki.ai), section
 * "FlashAttention-3": the transform is random signs followed by a Hadamard transform,
 * applied to queries and keys alike, so their dot products are unchanged in real
 * arithmetic while outliers are spread over all channels).  These functions define the
 * quantized inputs; the attention over them is the plain definition above, applied to
 * the dequantized values (code x scale).
 *
 * Readings where the pages leave a step open:
 *   - Q and K: each row is multiplied by the signs s (+1/-1 per channel) and by the
 *     Sylvester Hadamard matrix H_d (entries +-1) -- the unnormalised rotation, computed
 *     in fp32 by the butterfly below -- then quantized with one scale per block of 128
 *     rows of one head.  The dequantization scale carries 1/sqrt(d), which makes the
 *     rotation orthogonal: (x s H / sqrt(d)) . (y s H / sqrt(d)) = x . y.
 *   - V is not rotated (P V has no partner product to cancel a rotation) and gets one
 *     scale per (head, channel), which factors out of P V exactly.
 *   - Scales come from the block's largest magnitude: the largest element maps to 448,
 *     the largest finite e4m3 value.
 * Floating-point steps that decide a code are done in fp32 in a fixed order, so the
 * codes are a definite function of the inputs (bit-exact comparisons are possible).
 */

/* e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
 * Exponent field e >= 1: (1 + m/8) * 2^(e-7); e = 0: (m/8) * 2^-6 (subnormal). */
double oracle_e4m3_decode(int code) {
    const int sign = (code >> 7) & 1;
    const int e = (code >> 3) & 0xF;
    const int m = code & 7;
    if (e == 0xF && m == 7) return NAN;
    const double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 value, ties to the even code (mantissa bit 0 clear), magnitudes beyond
 * 448 saturate to 448; the sign of zero is kept.  Plain search over the 127 finite
 * non-negative codes, which increase with the code. */
int oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    const int sign = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    int lo = 0;
    for (int c = 1; c <= 0x7E; ++c)
        if (oracle_e4m3_decode(c) <= a) lo = c;
    if (lo == 0x7E) return sign | 0x7E;
    const double vlo = oracle_e4m3_decode(lo), vhi = oracle_e4m3_decode(lo + 1);
    const double mid = 0.5 * (vlo + vhi);
    int c;
    if (a < mid) c = lo;
    else if (a > mid) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;
    return sign | c;
}

/* x <- x H_d, unnormalised, in fp32, in place (d a power of two).  Stage h = 1, 2, 4,
 * ..., d/2 replaces the pair (x[i], x[i+h]) for each i with bit h clear by
 * (x[i] + x[i+h], x[i] - x[i+h]). */
static void fwht_f32(float* x, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; ++i)
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/* Q or K: x [heads, N, d] (values of the 16-bit inputs, exactly widened to fp32).
 * signs: d entries of +1/-1, or NULL for no rotation (per-block quantization only).
 * Outputs codes [heads, N, d] and scales [heads, ceil(N/128)]:
 *   y = x * s then y <- y H_d                     (if rotating)
 *   amax = max |y| over the block's rows and channels
 *   code = e4m3(y * (448 / amax))                 (fp32 division, then fp32 product)
 *   scale = amax * c, c = fl32(1 / (448 sqrt(d))) rotating, fl32(1 / 448) not
 * A block whose values are all zero gets scale 0 and codes e4m3(+-0). */
int oracle_fp8_quantize_qk(const float* x, const signed char* signs, int heads, int N, int d,
                           unsigned char* codes, float* scales) {
    if (heads <= 0 || N <= 0 || d <= 0 || (d & (d - 1)) != 0 || !x || !codes || !scales)
        return ORACLE_EINVAL;
    const int T = (N + 127) / 128;
    const float cfac = signs ? (float)(1.0 / (448.0 * sqrt((double)d))) : (float)(1.0 / 448.0);
    int failed = 0;
#pragma omp parallel
    {
        float* y = (float*)malloc(sizeof(float) * (size_t)128 * d);
        if (!y) {
#pragma omp atomic write
            failed = 1;
        }
        /* blocks are independent: the same result for any thread count */
#pragma omp for schedule(dynamic, 1)
        for (long ht = 0; ht < (long)heads * T; ++ht) {
            if (!y) continue;
            const int h = (int)(ht / T), t = (int)(ht % T);
            const int r0 = t * 128, r1 = (r0 + 128 < N) ? r0 + 128 : N;
            float amax = 0.f;
            for (int r = r0; r < r1; ++r) {
                float* yr = y + (size_t)(r - r0) * d;
                const float* xr = x + ((size_t)h * N + r) * d;
                for (int c = 0; c < d; ++c) yr[c] = (signs && signs[c] < 0) ? -xr[c] : xr[c];
                if (signs) fwht_f32(yr, d);
                for (int c = 0; c < d; ++c)
                    if (fabsf(yr[c]) > amax) amax = fabsf(yr[c]);
            }
            const float f = amax > 0.f ? 448.0f / amax : 0.f;
            scales[(size_t)h * T + t] = amax * cfac;
            for (int r = r0; r < r1; ++r)
                for (int c = 0; c < d; ++c)
                    codes[((size_t)h * N + r) * d + c] =
                        (unsigned char)oracle_e4m3_encode(y[(size_t)(r - r0) * d + c] * f);
        }
        free(y);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* V: v [heads, N, d].  One scale per (head, channel):
 *   amax_c = max over the head's N rows of |v_rc|
 *   code = e4m3(v * (448 / amax_c)),  scale_c = amax_c * fl32(1/448)
 * Outputs codes [heads, N, d] and scales [heads, d]. */
int oracle_fp8_quantize_v(const float* v, int heads, int N, int d, unsigned char* codes,
                          float* scales) {
    if (heads <= 0 || N <= 0 || d <= 0 || !v || !codes || !scales) return ORACLE_EINVAL;
    const float cfac = (float)(1.0 / 448.0);
    /* (head, channel) pairs are independent: the same result for any thread count */
#pragma omp parallel for schedule(dynamic, 1)
    for (long hc = 0; hc < (long)heads * d; ++hc) {
        const int h = (int)(hc / d), c = (int)(hc % d);
        float amax = 0.f;
        for (int r = 0; r < N; ++r) {
            const float a = fabsf(v[((size_t)h * N + r) * d + c]);
            if (a > amax) amax = a;
        }
        const float f = amax > 0.f ? 448.0f / amax : 0.f;
        scales[(size_t)h * d + c] = amax * cfac;
        for (int r = 0; r < N; ++r) {
            const size_t e = ((size_t)h * N + r) * d + c;
            codes[e] = (unsigned char)oracle_e4m3_encode(v[e] * f);
        }
    }
    return ORACLE_OK;
}

/* Element-wise front ends of the two functions above, for arrays. */
int oracle_e4m3_encode_array(const float* x, unsigned char* out, long n) {
    if (n < 0 || (n > 0 && (!x || !out))) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) out[i] = (unsigned char)oracle_e4m3_encode(x[i]);
    return ORACLE_OK;
}

int oracle_e4m3_decode_array(const unsigned char* c, double* out, long n) {
    if (n < 0 || (n > 0 && (!c || !out))) return ORACLE_EINVAL;
    for (long i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
    return ORACLE_OK;
}
