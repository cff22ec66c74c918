/*
 * gqa_oracle.c -- plain float64 CPU oracle for causal grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  It shares no code, header,
 * table or helper with the CUDA library, and the library never calls it.
 *
 * What it computes (written from the definition, slowly and on purpose):
 *
 *   "nx_f32_gqa_gate.nx source", header comment and tests T0-T5:
 *     scores = Q.K^T / sqrt(d); causal mask (token i attends only to j <= i);
 *     softmax; out = attn.V; H query heads share G < H key/value heads and
 *     query head h reads kv head h / (H/G)  (test T2).
 *     Backward of softmax: ds_j = a_j * (g_j - sum_k a_k g_k)   (test T4).
 *   "SnapKitty Transformer 8B", sections "FlashAttention Inference" and
 *   "Protected Inventions": the attention call takes causal, a sliding window
 *   and a number of attention sinks; the backward recomputes the
 *   probabilities from saved row statistics and uses D = rowsum(dO * O).
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of the repository):
 *   - window W > 0: query i sees key j when i - W < j <= i, plus every key
 *     j < n_sink with j <= i (the always-visible leading sink tokens).
 *     W <= 0 means no window and then n_sink is ignored.
 *   - causal == 0 means full attention (no window allowed).
 *   - scale is passed in by the caller (1/sqrt(d) by convention).
 *   - LSE_i = m_i + ln(l_i), the natural log of the sum of exp of the
 *     scaled scores.
 *
 * Layouts (all row-major, float64, exact widenings of the bf16 inputs):
 *   q, o, dO, dq : [B][H][S][d]      k, v, dk, dv : [B][G][S][d]
 *   lse          : [B][H][S]
 * Parity status: every function here is pinned by tests that do not call it
 * to check itself (worked example of page 5, closed forms, finite
 * differences, a library SDPA cross-check, literal mask sets).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The mask, exactly as read above.  Returns 1 when query i may see key j. */
int oracle_visible(long i, long j, int causal, int window, int n_sink)
{
    if (causal && j > i)
        return 0;
    if (causal && window > 0) {
        int in_window = (j > i - (long)window);
        int is_sink = (j < (long)n_sink);
        if (!in_window && !is_sink)
            return 0;
    }
    return 1;
}

/* One query row: fills p[0..S) with the attention weights of row i (zero where
 * masked), and returns LSE_i.  k and v point at the kv head this query head
 * reads.  s is scratch of length S. */
static double attention_row(const double *qi, const double *kg, int S, int d, long i,
                            int causal, int window, int n_sink, double scale,
                            double *s, double *p)
{
    double m = -INFINITY;
    for (long j = 0; j < S; ++j) {
        if (!oracle_visible(i, j, causal, window, n_sink)) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += qi[c] * kg[j * (long)d + c];
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    if (m == -INFINITY) {           /* no visible key: cannot happen under causal */
        for (long j = 0; j < S; ++j)
            p[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (long j = 0; j < S; ++j) {
        p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        l += p[j];
    }
    for (long j = 0; j < S; ++j)
        p[j] /= l;
    return m + log(l);
}

/* Forward over every (b, h, i).  o: [B][H][S][d], lse: [B][H][S]. */
void oracle_attn_fwd(const double *q, const double *k, const double *v,
                     double *o, double *lse,
                     int B, int H, int G, int S, int d,
                     int causal, int window, int n_sink, double scale)
{
    const int R = H / G;                       /* query heads per kv head */
    const long nrows = (long)B * H * S;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        double *p = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < nrows; ++r) {
            long i = r % S;
            long bh = r / S;
            int h = (int)(bh % H);
            int b = (int)(bh / H);
            int g = h / R;                          /* page 5, test T2 */
            const double *qi = q + r * d;
            const double *kg = k + ((long)b * G + g) * (long)S * d;
            const double *vg = v + ((long)b * G + g) * (long)S * d;
            double L = attention_row(qi, kg, S, d, i, causal, window, n_sink, scale, s, p);
            double *oi = o + r * d;
            for (int c = 0; c < d; ++c)
                oi[c] = 0.0;
            for (long j = 0; j < S; ++j) {
                if (p[j] == 0.0)
                    continue;
                for (int c = 0; c < d; ++c)
                    oi[c] += p[j] * vg[j * (long)d + c];
            }
            lse[r] = L;
        }
        free(s);
        free(p);
    }
}

/* Forward on a list of rows only: rows[3*n] = (b, h, i) triples.
 * o_rows: [n][d], lse_rows: [n].  Used to check full-size outputs by sampling. */
void oracle_attn_fwd_rows(const double *q, const double *k, const double *v,
                          double *o_rows, double *lse_rows,
                          int B, int H, int G, int S, int d,
                          int causal, int window, int n_sink, double scale,
                          const long *rows, int n)
{
    const int R = H / G;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        double *p = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < n; ++t) {
            long b = rows[3 * t], h = rows[3 * t + 1], i = rows[3 * t + 2];
            long g = h / R;
            const double *qi = q + ((b * H + h) * (long)S + i) * d;
            const double *kg = k + (b * G + g) * (long)S * d;
            const double *vg = v + (b * G + g) * (long)S * d;
            lse_rows[t] = attention_row(qi, kg, S, d, i, causal, window, n_sink, scale, s, p);
            double *oi = o_rows + (long)t * d;
            for (int c = 0; c < d; ++c)
                oi[c] = 0.0;
            for (long j = 0; j < S; ++j) {
                if (p[j] == 0.0)
                    continue;
                for (int c = 0; c < d; ++c)
                    oi[c] += p[j] * vg[j * (long)d + c];
            }
        }
        free(s);
        free(p);
    }
}

/* Backward of one kv group (b, g): the R query heads h = g*R .. g*R+R-1,
 * restricted to query rows i_begin <= i < i_end (all rows: 0 .. S).
 *   dq_g : [R][S][d]   gradients of those query heads (rows in range only)
 *   dk_g, dv_g : [S][d] gradients of kv head g from the rows in range
 * For each query row (exact P from its own forward, never a saved O/LSE):
 *   dP_ij = dO_i . v_j ;  D_i = sum_j P_ij dP_ij ;  dS_ij = P_ij (dP_ij - D_i)
 *   dq_i  = scale * sum_j dS_ij k_j
 *   dk_j += scale * dS_ij q_i ;  dv_j += P_ij dO_i       (summed over the group)
 * Rows are spread over threads; each thread keeps private dk/dv sums that are
 * added into the outputs one thread at a time at the end (float64, so the
 * order of those few additions does not matter at the tolerances used). */
void oracle_attn_bwd_group_rows(const double *q, const double *k, const double *v,
                                const double *dO, double *dq_g, double *dk_g, double *dv_g,
                                int B, int H, int G, int S, int d,
                                int causal, int window, int n_sink, double scale,
                                int b, int g, long i_begin, long i_end)
{
    (void)B;
    const int R = H / G;
    const double *kg = k + ((long)b * G + g) * (long)S * d;
    const double *vg = v + ((long)b * G + g) * (long)S * d;
    const long sd = (long)S * d;
    memset(dk_g, 0, sizeof(double) * sd);
    memset(dv_g, 0, sizeof(double) * sd);
    if (i_begin < 0)
        i_begin = 0;
    if (i_end > S)
        i_end = S;
    const long span = i_end > i_begin ? i_end - i_begin : 0;
    const long nrows = (long)R * span;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        double *p = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        double *dp = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        double *dk_t = (double *)calloc(sd > 0 ? sd : 1, sizeof(double));
        double *dv_t = (double *)calloc(sd > 0 ? sd : 1, sizeof(double));
#pragma omp for schedule(dynamic, 8)
        for (long r = 0; r < nrows; ++r) {
            int hh = (int)(r / span);
            long i = i_begin + r % span;
            int h = g * R + hh;
            const double *qi = q + (((long)b * H + h) * S + i) * d;
            const double *doi = dO + (((long)b * H + h) * S + i) * d;
            attention_row(qi, kg, S, d, i, causal, window, n_sink, scale, s, p);
            double D = 0.0;
            for (long j = 0; j < S; ++j) {
                dp[j] = 0.0;
                if (p[j] == 0.0)
                    continue;
                for (int c = 0; c < d; ++c)
                    dp[j] += doi[c] * vg[j * (long)d + c];
                D += p[j] * dp[j];
            }
            double *dqi = dq_g + ((long)hh * S + i) * d;
            for (int c = 0; c < d; ++c)
                dqi[c] = 0.0;
            for (long j = 0; j < S; ++j) {
                if (p[j] == 0.0)
                    continue;
                double ds = p[j] * (dp[j] - D);
                for (int c = 0; c < d; ++c) {
                    dqi[c] += scale * ds * kg[j * (long)d + c];
                    dk_t[j * (long)d + c] += scale * ds * qi[c];
                    dv_t[j * (long)d + c] += p[j] * doi[c];
                }
            }
        }
#pragma omp critical
        {
            for (long e = 0; e < sd; ++e) {
                dk_g[e] += dk_t[e];
                dv_g[e] += dv_t[e];
            }
        }
        free(s);
        free(p);
        free(dp);
        free(dk_t);
        free(dv_t);
    }
}

/* Whole group: every query row of its R heads. */
void oracle_attn_bwd_group(const double *q, const double *k, const double *v, const double *dO,
                           double *dq_g, double *dk_g, double *dv_g,
                           int B, int H, int G, int S, int d,
                           int causal, int window, int n_sink, double scale,
                           int b, int g)
{
    oracle_attn_bwd_group_rows(q, k, v, dO, dq_g, dk_g, dv_g, B, H, G, S, d,
                               causal, window, n_sink, scale, b, g, 0, S);
}

/* Threads the OpenMP runtime will use (reported with CPU timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Backward over every group.  dq: [B][H][S][d], dk, dv: [B][G][S][d]. */
void oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dO,
                     double *dq, double *dk, double *dv,
                     int B, int H, int G, int S, int d,
                     int causal, int window, int n_sink, double scale)
{
    const int R = H / G;
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < G; ++g)
            oracle_attn_bwd_group(q, k, v, dO,
                                  dq + (((long)b * H + (long)g * R) * S) * d,
                                  dk + (((long)b * G + g) * (long)S) * d,
                                  dv + (((long)b * G + g) * (long)S) * d,
                                  B, H, G, S, d, causal, window, n_sink, scale, b, g);
}

/* ------------------------------------------------------------------ YaRN RoPE
 *
 * "SnapKitty Transformer 8B" (model specification table and section
 * "Protected Inventions") applies YaRN-scaled rotary position embeddings with
 * a 32x factor for 204800-token sequences to the queries and keys.  The pages
 * give no formula; the definition written out here is the published one:
 * "YaRN: Efficient Context Window Extension of Large Language Models" (Peng,
 * Quesnelle, Fan, Shippole, 2023), section 3 ("NTK-by-parts" interpolation and
 * the attention temperature), on rotary embeddings as defined by RoFormer
 * (Su et al.): dimension pair i = (2i, 2i+1) of a row at position m is turned
 * by the angle m * h_i.
 *
 *   theta_i   = base^(-2i/d)                 wavelength lambda_i = 2 pi / theta_i
 *   r_i       = L / lambda_i                 (L: the original context length)
 *   gamma(r)  = 0 if r < alpha, 1 if r > beta, (r - alpha) / (beta - alpha) else
 *   h_i       = (1 - gamma(r_i)) theta_i / s + gamma(r_i) theta_i     (s: factor)
 *   sqrt(1/t) = 0.1 ln(s) + 1                (attention temperature; the logits
 *                                             are multiplied by 1/t)
 */
void oracle_yarn_freqs(int d, double base, double factor, double orig_ctx, double alpha,
                       double beta, double *freq)
{
    for (int i = 0; i < d / 2; ++i) {
        double theta = pow(base, -2.0 * i / d);
        double wavelength = 2.0 * acos(-1.0) / theta;   /* 2 pi / theta */
        double r = orig_ctx / wavelength;
        double gamma;
        if (r < alpha)
            gamma = 0.0;
        else if (r > beta)
            gamma = 1.0;
        else
            gamma = (r - alpha) / (beta - alpha);
        freq[i] = (1.0 - gamma) * theta / factor + gamma * theta;
    }
}

/* sqrt(1/t) of the attention temperature for scale factor s. */
double oracle_yarn_mscale(double factor)
{
    return 0.1 * log(factor) + 1.0;
}

/* Rotates n rows of x ([n][d]) to out: row r sits at position pos[r]. */
void oracle_rope_rotate(const double *x, double *out, const long *pos, long n, int d,
                        const double *freq)
{
    for (long r = 0; r < n; ++r) {
        for (int i = 0; i < d / 2; ++i) {
            double a = (double)pos[r] * freq[i];
            double c = cos(a), s = sin(a);
            double x0 = x[r * d + 2 * i], x1 = x[r * d + 2 * i + 1];
            out[r * d + 2 * i] = x0 * c - x1 * s;
            out[r * d + 2 * i + 1] = x0 * s + x1 * c;
        }
    }
}

/* Rounds each value to the nearest bf16 (ties to even) by way of fp32: the
 * rotated queries and keys are bf16 tensors in a bf16 model, so the attention
 * that follows the rotation sees them rounded once.  n values in place. */
void oracle_round_bf16(double *x, long n)
{
    for (long e = 0; e < n; ++e) {
        float f = (float)x[e];
        unsigned int u;
        memcpy(&u, &f, sizeof u);
        if ((u & 0x7f800000u) != 0x7f800000u) {      /* finite: round the low 16 bits */
            u += 0x7fffu + ((u >> 16) & 1u);
        }
        u &= 0xffff0000u;
        memcpy(&f, &u, sizeof f);
        x[e] = (double)f;
    }
}

/* ---------------------------------------------------------------- FP8 E4M3
 *
 * "SnapKitty Transformer 8B" (section "Protected Inventions") names a forward
 * "with FP8 computation"; the pages give no format.  The format taken is the
 * OCP 8-bit floating point specification's E4M3 (the fp8 type of the sm_100
 * tensor cores): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 encodes subnormals m / 8 * 2^-6; S.1111.111 is NaN and
 * there are no infinities (largest finite value 448).  A tensor is stored as
 * bytes plus one fp32 scale: value = decode(byte) * scale.  The oracle takes
 * those exact values and runs the float64 definition on them.
 */
double oracle_decode_e4m3(unsigned char b)
{
    int sign = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* out[i] = decode(bytes[i]) * scale for n values. */
void oracle_decode_e4m3_array(const unsigned char *bytes, double *out, long n, double scale)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_decode_e4m3(bytes[i]) * scale;
}
