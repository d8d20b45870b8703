/*
 * gdn_oracle.c -- plain, slow fp64 CPU oracle for the gated-delta SSM layer step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file: only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or helper with the CUDA
 * kernels; the two meet only at the seeded inputs.
 *
 * Every value is widened to double on entry and all arithmetic is double.
 * Inputs arrive as float32 arrays: bf16 and fp32 activations are both exactly
 * representable there, so the oracle sees the very values the GPU sees.
 * Build with -O2 -fno-fast-math -ffp-contract=off so each line computes what
 * it says.
 *
 * Sources (the web pages this layer is specified on):
 *   [hdr]  "fm_kernel_ssm.h" (Foundry Metal kernel family for the gated-delta
 *          SSM): sections "Decay gate", "Causal depthwise conv1d + SiLU",
 *          "Gated RMSNorm", "Delta-rule recurrence".
 *   [rs]   "ssm_mamba.rs" (spark_model layer ops): doc comments of
 *          conv1d_update_l2norm (SiLU then per-head L2 norm on the Q/K
 *          channels only) and gdn_verify_fused_conv_k2 (K=2 verify with a
 *          position-0 rollback snapshot).
 *   [scr]  "scr_state.hpp": the "GDN staleness" comment and log_gate (the
 *          guarded softplus, the L2 form k = cv / sqrt(sum cv^2 + eps), and the
 *          matrix form S' = g (I - b k k^T) S + b k v^T).
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - V head h reads QK head floor(h / r), r = Hv / Hq ("GQA-repeated").
 *   - decay is applied before the prediction, the readout uses the updated
 *     state, scale = 1/sqrt(d_k).
 *   - conv history is [conv_dim][W-1], oldest first; no conv bias.
 *
 * Parity pins: every function here is pinned by the CPU tests (closed forms,
 * library routines, brute-force matrix form, invariants). The composition of
 * the whole layer has no worked numeric example on the pages and is pinned
 * only through its parts: "parity unpinned" for the composed layer beyond
 * those pins.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* softplus guarded at 20: above 20 it is the identity ([hdr] "Decay gate";
 * [scr] log_gate uses the same strict v > 20 test). */
double gdnref_softplus(double v)
{
    if (v > 20.0)
        return v;
    return log1p(exp(v));
}

double gdnref_sigmoid(double v)
{
    return 1.0 / (1.0 + exp(-v));
}

double gdnref_silu(double v)
{
    return v * gdnref_sigmoid(v);
}

/* g[r][h] = a[h] * softplus(alpha[r][h] + dt[h]) with a[h] = -exp(A_log[h]);
 * g is left pre-exp ([hdr] "Decay gate"; [scr] log_gate). */
void gdnref_decay_gate(const float *alpha, const float *dt, const float *A_log,
                       double *g, long rows, int n_heads)
{
    for (long r = 0; r < rows; ++r) {
        for (int h = 0; h < n_heads; ++h) {
            double a = -exp((double)A_log[h]);
            double v = (double)alpha[r * n_heads + h] + (double)dt[h];
            g[r * n_heads + h] = a * gdnref_softplus(v);
        }
    }
}

/* One token of the depthwise causal conv1d + SiLU over conv_dim channels
 * ([hdr] "Causal depthwise conv1d + SiLU"). Channel c's window is
 * [hist[c][0] .. hist[c][W-2], x[c]] against taps w[c][0..W-1]; the history
 * then drops its oldest entry and appends the RAW input x[c]. */
void gdnref_conv_step(const float *x, const float *w, double *hist, double *out,
                      int conv_dim, int W)
{
    for (int c = 0; c < conv_dim; ++c) {
        double *hc = hist + (size_t)c * (W - 1);
        const float *wc = w + (size_t)c * W;
        double acc = 0.0;
        for (int t = 0; t < W - 1; ++t)
            acc += hc[t] * (double)wc[t];
        acc += (double)x[c] * (double)wc[W - 1];
        out[c] = gdnref_silu(acc);
        for (int t = 0; t + 1 < W - 1; ++t)
            hc[t] = hc[t + 1];
        if (W > 1)
            hc[W - 2] = (double)x[c];
    }
}

/* v <- v / sqrt(sum v^2 + eps) ([scr] "GDN staleness": k = cv / sqrt(sum cv^2 + eps);
 * [rs] conv1d_update_l2norm: applied per head to the Q and K channels). */
void gdnref_l2norm(double *v, int n, double eps)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i)
        s += v[i] * v[i];
    double inv = 1.0 / sqrt(s + eps);
    for (int i = 0; i < n; ++i)
        v[i] = v[i] * inv;
}

/* One decode step for one head in the plain orientation S[i][j] (i = key
 * index, j = value index), written from [hdr] "Delta-rule recurrence":
 *   S <- exp(g) S                      decay
 *   pred_j = sum_i S[i][j] k[i]        prediction with the decayed state
 *   u_j = beta (v_j - pred_j)          delta
 *   S[i][j] += k[i] u_j                rank-1 write
 *   o_j = scale * sum_i S[i][j] q[i]   readout of the UPDATED state
 */
void gdnref_recurrence_step(double *S, const double *q, const double *k,
                            const double *v, double g, double beta, double *o,
                            int d, double scale)
{
    double decay = exp(g);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(size_t)i * d + j] *= decay;
    double *u = (double *)malloc(sizeof(double) * (size_t)d);
    for (int j = 0; j < d; ++j) {
        double pred = 0.0;
        for (int i = 0; i < d; ++i)
            pred += S[(size_t)i * d + j] * k[i];
        u[j] = beta * (v[j] - pred);
    }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(size_t)i * d + j] += k[i] * u[j];
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += S[(size_t)i * d + j] * q[i];
        o[j] = scale * acc;
    }
    free(u);
}

/* Per-head gated RMSNorm ([hdr] "Gated RMSNorm"):
 *   inv = 1 / sqrt(mean(y^2) + eps);  out = ((y * inv) * w) * silu(z)
 * w has head_dim entries and is shared by every head. */
void gdnref_gated_norm(const double *y, const float *w, const double *z,
                       double *out, int d, double eps)
{
    double ss = 0.0;
    for (int j = 0; j < d; ++j)
        ss += y[j] * y[j];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int j = 0; j < d; ++j)
        out[j] = ((y[j] * inv) * (double)w[j]) * gdnref_silu(z[j]);
}

/*
 * Round a double to the nearest bfloat16 value, ties to even: the storage
 * rounding of the bf16-state decode variant (a serving option that has no
 * counterpart on the pages). bfloat16 keeps float32's exponent range and 8
 * significant bits, so a value in the binade [2^(e-1), 2^e) is rounded to a
 * multiple of 2^(e-8); below 2^-126 the spacing stays 2^-133 (subnormals);
 * a result of magnitude 2^128 or more is an overflow to infinity.
 */
double gdnref_round_bf16(double v)
{
    if (v != v || v == 0.0 || isinf(v))
        return v;
    int e;
    frexp(v, &e);
    int q = e - 8;
    if (q < -133)
        q = -133;
    /* scaling by a power of two is exact; rint rounds half to even */
    const double r = ldexp(rint(ldexp(v, -q)), q);
    if (fabs(r) >= ldexp(1.0, 128))
        return v > 0 ? INFINITY : -INFINITY;
    return r;
}

/*
 * The whole layer step for ONE sequence over T tokens, one token at a time.
 *
 * Per token: conv + SiLU over all channels; split [Q | K | V]; L2-normalise
 * each Q head and each K head; gates g (pre-exp) and beta = sigmoid(logit)
 * per V head; the recurrence for each V head against QK head h / r; gated
 * RMSNorm per V head.
 *
 * Layouts (row strides in elements):
 *   x      [T][x_stride]  first conv_dim entries = Q | K | V, conv_dim = (2 Hq + Hv) d
 *   z      [T][z_stride]  first Hv*d entries
 *   alpha, beta_logit [T][Hv]
 *   conv_w [conv_dim][W], dt/A_log [Hv], norm_w [d]
 *   S      [Hv][d][d] plain orientation S[h][i][j], updated in place
 *   hist   [conv_dim][W-1] oldest first, updated in place
 *   out    [T][Hv][d]
 * Optional (NULL to skip):
 *   conv_out [T][conv_dim]  post-SiLU, Q/K post-L2
 *   g_out, beta_out [T][Hv]
 *   y_out  [T][Hv][d]       recurrence readout before the norm
 *   snap_after >= 0: after that token, S and hist are copied to S_snap/hist_snap.
 * bf16_state != 0: the bf16-state variant. After each head's step (whose
 * readout uses the updated state before rounding) its state is rounded to
 * bfloat16, and each output value is rounded to bfloat16.
 * Returns 0, or -1 on a bad shape.
 */
int gdnref_layer(int T, int Hq, int Hv, int d, int W,
                 const float *x, long x_stride,
                 const float *z, long z_stride,
                 const float *alpha, const float *beta_logit,
                 const float *conv_w, const float *dt, const float *A_log,
                 const float *norm_w, double l2_eps, double rms_eps,
                 double *S, double *hist, double *out,
                 double *conv_out, double *g_out, double *beta_out, double *y_out,
                 int snap_after, double *S_snap, double *hist_snap, int bf16_state)
{
    if (T < 0 || Hq <= 0 || Hv <= 0 || d <= 0 || W < 1 || Hv % Hq != 0)
        return -1;
    const int r = Hv / Hq;
    const int conv_dim = (2 * Hq + Hv) * d;
    const double scale = 1.0 / sqrt((double)d);
    double *c = (double *)malloc(sizeof(double) * (size_t)conv_dim);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    double *zz = (double *)malloc(sizeof(double) * (size_t)d);
    double *g = (double *)malloc(sizeof(double) * (size_t)Hv);
    if (!c || !y || !zz || !g) {
        free(c); free(y); free(zz); free(g);
        return -1;
    }
    for (int t = 0; t < T; ++t) {
        gdnref_conv_step(x + (size_t)t * x_stride, conv_w, hist, c, conv_dim, W);
        double *qs = c;
        double *ks = c + (size_t)Hq * d;
        double *vs = c + (size_t)2 * Hq * d;
        for (int h = 0; h < Hq; ++h) {
            gdnref_l2norm(qs + (size_t)h * d, d, l2_eps);
            gdnref_l2norm(ks + (size_t)h * d, d, l2_eps);
        }
        gdnref_decay_gate(alpha + (size_t)t * Hv, dt, A_log, g, 1, Hv);
        if (conv_out)
            memcpy(conv_out + (size_t)t * conv_dim, c, sizeof(double) * (size_t)conv_dim);
        for (int h = 0; h < Hv; ++h) {
            int hk = h / r;
            double beta = gdnref_sigmoid((double)beta_logit[(size_t)t * Hv + h]);
            if (g_out)
                g_out[(size_t)t * Hv + h] = g[h];
            if (beta_out)
                beta_out[(size_t)t * Hv + h] = beta;
            gdnref_recurrence_step(S + (size_t)h * d * d, qs + (size_t)hk * d,
                                   ks + (size_t)hk * d, vs + (size_t)h * d,
                                   g[h], beta, y, d, scale);
            if (y_out)
                memcpy(y_out + ((size_t)t * Hv + h) * d, y, sizeof(double) * (size_t)d);
            const float *zt = z + (size_t)t * z_stride + (size_t)h * d;
            for (int j = 0; j < d; ++j)
                zz[j] = (double)zt[j];
            double *oh = out + ((size_t)t * Hv + h) * d;
            gdnref_gated_norm(y, norm_w, zz, oh, d, rms_eps);
            if (bf16_state) {
                double *Sh = S + (size_t)h * d * d;
                for (size_t e = 0; e < (size_t)d * d; ++e)
                    Sh[e] = gdnref_round_bf16(Sh[e]);
                for (int j = 0; j < d; ++j)
                    oh[j] = gdnref_round_bf16(oh[j]);
            }
        }
        if (t == snap_after) {
            if (S_snap)
                memcpy(S_snap, S, sizeof(double) * (size_t)Hv * d * d);
            if (hist_snap)
                memcpy(hist_snap, hist, sizeof(double) * (size_t)conv_dim * (W - 1));
        }
    }
    free(c); free(y); free(zz); free(g);
    return 0;
}

/*
 * The recurrence alone, scanned over T tokens for ONE head, from already
 * prepared inputs (q, k normalised; beta already a sigmoid; g pre-exp):
 * the sequential scan the chunked prefill is held to ([hdr] "Delta-rule
 * recurrence", the sequential-scan entry kept as the permanent reference).
 *   q, k, v [T][d], g, beta [T], S [d][d] plain orientation, y [T][d].
 */
void gdnref_recurrence_scan(int T, int d, const double *q, const double *k,
                            const double *v, const double *g, const double *beta,
                            double *S, double *y, double scale)
{
    for (int t = 0; t < T; ++t)
        gdnref_recurrence_step(S, q + (size_t)t * d, k + (size_t)t * d,
                               v + (size_t)t * d, g[t], beta[t],
                               y + (size_t)t * d, d, scale);
}
