/*
 * CPU oracle for the batch-invariant DiT AdaLN final modulation ("norm_out"),
 * forward and backward.
 *
 * TEST INFRASTRUCTURE.  This is a plain, slow, obviously-correct host
 * implementation used only to check the CUDA library: the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it, nothing else does.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared -lm
 * (no contraction into FMA, IEEE single/double arithmetic as written).
 *
 * What it computes (sources):
 *
 *  [op]    RL-Kernel PR 538 "final_adaln_out", section "What":
 *            scale, shift = (SiLU(temb) @ W^T + b).chunk(2)   (3072 -> 6144,
 *                                                              scale first)
 *            out = LayerNorm(x, eps=1e-6, no affine) * (1 + scale) + shift
 *          and the backward: dx, d_scale/d_shift as token sums, dW/db/d_temb.
 *  [round] miles_diffusion PR 108 "bitwise train<->rollout parity via
 *          autocast-parity norms and a pinned flash kernel", Summary, root
 *          cause 1 (and its second rendering, "Patches"): LayerNorm computes
 *          and returns fp32, (1 + scale) rounds once in bf16, the modulation
 *          promotes to fp32, one bf16 rounding at the store.
 *  [tree]  RL-Kernel PR 538, section "What" (token sums by a fixed 32-way
 *          balanced tree whose shape depends only on the sequence length) and
 *          the review thread on the cancellation case (each 32-token tile is
 *          summed in ascending order with Neumaier compensation; tile sums and
 *          corrections are folded level by level; one final IEEE add).
 *  [ref]   RL-Kernel PR 538, section "What": an independent CPU reference with
 *          sequential Neumaier token sums; review findings ask for a
 *          compensated input gradient and bias gradient as well.
 *
 * Every sum here is a sequential Neumaier sum in fp64 (compensated, so it is
 * correct to about one fp64 ulp), every product of two bf16 values or of a
 * bf16 and an fp32 value is exact in fp64, and the only roundings are the
 * ones the operator defines.  Readings of points the pages leave open:
 *
 *  - LayerNorm variance is the biased one (divide by D), eps = fp32(1e-6) is
 *    added to the variance inside the square root.
 *  - SiLU output u is the bf16 nearest to the fp64 value of t/(1+exp(-t))
 *    (the correctly rounded SiLU for every |t| >= 2^-125; below that the fp64
 *    value is t/2 and can sit on a bf16 tie).
 *  - The projection bias is added before the single bf16 rounding of emb.
 *  - onep = bf16(fp32(1 + scale)); m = fp32(fp32(xhat * onep) + shift), xhat
 *    being the fp32 rounding of the exact LayerNorm value; out = bf16(m).
 *  - d_scale[b,d] = sum_s g*xhat (xhat the fp32 forward value), d_shift[b,d]
 *    = sum_s g, g = fp32(dy); both returned in fp32.
 *  - dx = bf16(exact LayerNorm backward of g*onep).
 *  - The projection backward takes e = bf16(d_emb); d_temb = bf16(d_silu *
 *    silu'(t)); dW = sum_b e*u, db = sum_b e.
 *
 * The fp32 token tree (oracle_token_tree_f32) and the fp32 sequential weight
 * gradient (oracle_wgrad_seq_f32) replay the operator's own fixed orders in
 * fp32 from their definitions above, so that the library's results can be
 * checked bit for bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* number formats                                                            */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }
static double bf16_to_f64(uint16_t h) { return (double)bf16_to_f32(h); }

/* nearest bf16 to a float (ties to even) */
static uint16_t bf16_from_f32(float f)
{
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* nearest bf16 to a double (ties to even), rounded once, not through fp32 */
static uint16_t bf16_from_f64(double x)
{
    if (x != x) return 0x7FC0u;
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    double a = fabs(x);
    int e;
    frexp(a, &e);            /* a = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;           /* spacing of 8 significant bits */
    if (q < -133) q = -133;  /* bf16 subnormal spacing 2^-133 */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    float rf = (float)r;     /* exact (or overflow to inf) */
    uint16_t h = (uint16_t)(bits_from_f32(rf) >> 16);
    return x < 0 ? (uint16_t)(h | 0x8000u) : h;
}

/* ------------------------------------------------------------------------ */
/* compensated summation in fp64                                             */
/* ------------------------------------------------------------------------ */

typedef struct { double s, c; } nsum;

static void nsum_add(nsum *a, double v)
{
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
    else                       a->c += (v - t) + a->s;
    a->s = t;
}
static double nsum_val(const nsum *a) { return a->s + a->c; }

/* ------------------------------------------------------------------------ */
/* SiLU and its derivative, fp64                                             */
/* ------------------------------------------------------------------------ */

static double sigmoid64(double t) { return 1.0 / (1.0 + exp(-t)); }
static double silu64(double t) { return t * sigmoid64(t); }
/* d/dt [t * sigma(t)] = sigma(t) * (1 + t * (1 - sigma(t)))               */
static double dsilu64(double t) { double s = sigmoid64(t); return s * (1.0 + t * (1.0 - s)); }

void oracle_silu_bf16(const uint16_t *t, uint16_t *u, long n)
{
    for (long i = 0; i < n; ++i) u[i] = bf16_from_f64(silu64(bf16_to_f64(t[i])));
}

void oracle_dsilu_f64(const double *t, double *out, long n)
{
    for (long i = 0; i < n; ++i) out[i] = dsilu64(t[i]);
}

/* ------------------------------------------------------------------------ */
/* shared cores                                                              */
/* ------------------------------------------------------------------------ */

/* emb[b,n] = sum_k u[b,k] * W[n,k] + bias[n], compensated fp64, for the
 * output rows n0 <= n < n1 (emb keeps its row stride N)                    */
static void proj_core(const double *u, const double *W, const double *bias,
                      double *emb, int B, int K, int N, int n0, int n1)
{
    for (int b = 0; b < B; ++b)
        for (int n = n0; n < n1; ++n) {
            nsum acc = {0.0, 0.0};
            const double *w = W + (size_t)n * K;
            const double *ub = u + (size_t)b * K;
            for (int k = 0; k < K; ++k) nsum_add(&acc, ub[k] * w[k]);
            nsum_add(&acc, bias[n]);
            emb[(size_t)b * N + n] = nsum_val(&acc);
        }
}

/* LayerNorm of one row (no affine): biased variance, eps inside the sqrt */
static void ln_row(const double *x, int D, double eps, double *mu_out,
                   double *rstd_out, double *xhat)
{
    nsum s = {0.0, 0.0};
    for (int d = 0; d < D; ++d) nsum_add(&s, x[d]);
    double mu = nsum_val(&s) / D;
    nsum v = {0.0, 0.0};
    for (int d = 0; d < D; ++d) { double c = x[d] - mu; nsum_add(&v, c * c); }
    double var = nsum_val(&v) / D;
    double rstd = 1.0 / sqrt(var + eps);
    for (int d = 0; d < D; ++d) xhat[d] = (x[d] - mu) * rstd;
    *mu_out = mu;
    *rstd_out = rstd;
}

/* LayerNorm backward of one row: given the upstream gradient gh of the
 * normalised value, dx = rstd * (gh - mean(gh) - xhat * mean(gh * xhat)).   */
static void ln_bwd_row(const double *gh, const double *xhat, double rstd, int D,
                       double *dx)
{
    nsum s1 = {0.0, 0.0}, s2 = {0.0, 0.0};
    for (int d = 0; d < D; ++d) { nsum_add(&s1, gh[d]); nsum_add(&s2, gh[d] * xhat[d]); }
    double c1 = nsum_val(&s1) / D;
    double c2 = nsum_val(&s2) / D;
    for (int d = 0; d < D; ++d) dx[d] = rstd * (gh[d] - c1 - xhat[d] * c2);
}

/* ------------------------------------------------------------------------ */
/* projection forward                                                        */
/* ------------------------------------------------------------------------ */

/* emb = bf16( bf16(silu(temb)) @ W^T + b ); W is [2D, D] row-major,
 * emb [B, 2D] = [scale | shift].  Only the output rows n0 <= n < n1 are
 * written (oracle_proj_fwd: all of them).                                   */
void oracle_proj_fwd_rows(const uint16_t *temb, const uint16_t *W, const uint16_t *bias,
                          uint16_t *emb, int B, int D, int n0, int n1)
{
    int N = 2 * D;
    double *u = malloc(sizeof(double) * (size_t)B * D);
    double *w = malloc(sizeof(double) * (size_t)N * D);
    double *bb = malloc(sizeof(double) * (size_t)N);
    double *e = malloc(sizeof(double) * (size_t)B * N);
    for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = bf16_to_f64(bf16_from_f64(silu64(bf16_to_f64(temb[i]))));
    for (size_t i = (size_t)n0 * D; i < (size_t)n1 * D; ++i) w[i] = bf16_to_f64(W[i]);
    for (int n = n0; n < n1; ++n) bb[n] = bf16_to_f64(bias[n]);
    proj_core(u, w, bb, e, B, D, N, n0, n1);
    for (int b = 0; b < B; ++b)
        for (int n = n0; n < n1; ++n) emb[(size_t)b * N + n] = bf16_from_f64(e[(size_t)b * N + n]);
    free(u); free(w); free(bb); free(e);
}

void oracle_proj_fwd(const uint16_t *temb, const uint16_t *W, const uint16_t *bias,
                     uint16_t *emb, int B, int D)
{
    oracle_proj_fwd_rows(temb, W, bias, emb, B, D, 0, 2 * D);
}

/* the same map without any rounding */
void oracle_proj_fwd_f64(const double *temb, const double *W, const double *bias,
                         double *emb, int B, int D)
{
    int N = 2 * D;
    double *u = malloc(sizeof(double) * (size_t)B * D);
    for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = silu64(temb[i]);
    proj_core(u, W, bias, emb, B, D, N, 0, N);
    free(u);
}

/* ------------------------------------------------------------------------ */
/* LayerNorm + modulation forward                                            */
/* ------------------------------------------------------------------------ */

/* out = bf16( fp32( fp32(xhat * onep) + shift ) ), onep = bf16(fp32(1+scale)),
 * xhat = fp32(exact LayerNorm).  mean/rstd: fp32 roundings of the exact row
 * statistics (nullable).                                                     */
void oracle_out_fwd(const uint16_t *x, const uint16_t *emb, float eps, uint16_t *out,
                    float *mean, float *rstd, int B, int S, int D)
{
    double *xr = malloc(sizeof(double) * (size_t)D);
    double *xh = malloc(sizeof(double) * (size_t)D);
    float *onep = malloc(sizeof(float) * (size_t)D);
    float *shift = malloc(sizeof(float) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        const uint16_t *e = emb + (size_t)b * 2 * D;
        for (int d = 0; d < D; ++d) {
            onep[d] = bf16_to_f32(bf16_from_f32(1.0f + bf16_to_f32(e[d])));
            shift[d] = bf16_to_f32(e[D + d]);
        }
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            const uint16_t *xs = x + row * D;
            for (int d = 0; d < D; ++d) xr[d] = bf16_to_f64(xs[d]);
            double mu, r;
            ln_row(xr, D, (double)eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d) {
                float xf = (float)xh[d];
                float prod = xf * onep[d];
                float m = prod + shift[d];
                out[row * D + d] = bf16_from_f32(m);
            }
            if (mean) mean[row] = (float)mu;
            if (rstd) rstd[row] = (float)r;
        }
    }
    free(xr); free(xh); free(onep); free(shift);
}

/* out = LayerNorm(x) * (1 + scale) + shift, everything fp64, no rounding */
void oracle_out_fwd_f64(const double *x, const double *scale, const double *shift,
                        double eps, double *out, int B, int S, int D)
{
    double *xh = malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            double mu, r;
            ln_row(x + row * D, D, eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d)
                out[row * D + d] = xh[d] * (1.0 + scale[(size_t)b * D + d]) + shift[(size_t)b * D + d];
        }
    free(xh);
}

/* ------------------------------------------------------------------------ */
/* LayerNorm + modulation backward                                           */
/* ------------------------------------------------------------------------ */

/* dx = bf16(LayerNorm backward of g*onep), g = fp32(dy);
 * d_emb[b, 0:D]  = d_scale = sum_s g * xhat_f32,
 * d_emb[b, D:2D] = d_shift = sum_s g,
 * token sums sequential over s (ascending) with Neumaier compensation in
 * fp64, returned rounded to fp32.  xhat is recomputed from x.               */
void oracle_out_bwd(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, float eps,
                    uint16_t *dx, float *d_emb, int B, int S, int D)
{
    double *xr = malloc(sizeof(double) * (size_t)D);
    double *xh = malloc(sizeof(double) * (size_t)D);
    double *gh = malloc(sizeof(double) * (size_t)D);
    double *dxr = malloc(sizeof(double) * (size_t)D);
    double *onep = malloc(sizeof(double) * (size_t)D);
    nsum *ss = malloc(sizeof(nsum) * (size_t)D);
    nsum *sh = malloc(sizeof(nsum) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        const uint16_t *e = emb + (size_t)b * 2 * D;
        for (int d = 0; d < D; ++d) {
            onep[d] = (double)bf16_to_f32(bf16_from_f32(1.0f + bf16_to_f32(e[d])));
            ss[d].s = ss[d].c = 0.0;
            sh[d].s = sh[d].c = 0.0;
        }
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            for (int d = 0; d < D; ++d) xr[d] = bf16_to_f64(x[row * D + d]);
            double mu, r;
            ln_row(xr, D, (double)eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d) {
                double g = bf16_to_f64(dy[row * D + d]);
                gh[d] = g * onep[d];                   /* exact */
                nsum_add(&ss[d], g * (double)(float)xh[d]); /* exact product */
                nsum_add(&sh[d], g);
            }
            ln_bwd_row(gh, xh, r, D, dxr);
            for (int d = 0; d < D; ++d) dx[row * D + d] = bf16_from_f64(dxr[d]);
        }
        for (int d = 0; d < D; ++d) {
            d_emb[(size_t)b * 2 * D + d] = (float)nsum_val(&ss[d]);
            d_emb[(size_t)b * 2 * D + D + d] = (float)nsum_val(&sh[d]);
        }
    }
    free(xr); free(xh); free(gh); free(dxr); free(onep); free(ss); free(sh);
}

/* exact gradients of oracle_out_fwd_f64 for upstream gradient dy */
void oracle_out_bwd_f64(const double *dy, const double *x, const double *scale, double eps,
                        double *dx, double *d_scale, double *d_shift, int B, int S, int D)
{
    double *xh = malloc(sizeof(double) * (size_t)D);
    double *gh = malloc(sizeof(double) * (size_t)D);
    nsum *ss = malloc(sizeof(nsum) * (size_t)D);
    nsum *sh = malloc(sizeof(nsum) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        for (int d = 0; d < D; ++d) { ss[d].s = ss[d].c = 0.0; sh[d].s = sh[d].c = 0.0; }
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            double mu, r;
            ln_row(x + row * D, D, eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d) {
                double g = dy[row * D + d];
                gh[d] = g * (1.0 + scale[(size_t)b * D + d]);
                nsum_add(&ss[d], g * xh[d]);
                nsum_add(&sh[d], g);
            }
            ln_bwd_row(gh, xh, r, D, dx + row * D);
        }
        for (int d = 0; d < D; ++d) {
            d_scale[(size_t)b * D + d] = nsum_val(&ss[d]);
            d_shift[(size_t)b * D + d] = nsum_val(&sh[d]);
        }
    }
    free(xh); free(gh); free(ss); free(sh);
}

/* ------------------------------------------------------------------------ */
/* token sums                                                                */
/* ------------------------------------------------------------------------ */

/* out[b,h] = sum_s in[b,s,h], sequential in s with Neumaier compensation (fp64) */
void oracle_token_sum_f64(const float *in, double *out, int B, int S, int H)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            nsum a = {0.0, 0.0};
            for (int s = 0; s < S; ++s) nsum_add(&a, (double)in[((size_t)b * S + s) * H + h]);
            out[(size_t)b * H + h] = nsum_val(&a);
        }
}

/* one Neumaier step in fp32: t = s + v; the part of the smaller operand lost
 * in t goes into the compensation c.  |s| == |v| takes the first branch.     */
static void nstep_f32(float *s, float *c, float v)
{
    float t = *s + v;
    float lost;
    if (fabsf(*s) >= fabsf(v)) { float d = *s - t; lost = d + v; }
    else                       { float d = v - t;  lost = d + *s; }
    *c = *c + lost;
    *s = t;
}

#define TREE_FAN 32

/* The fixed 32-way token tree, in fp32:
 *  level 0: tokens are cut into tiles of 32 (the last tile may be short);
 *           each tile is a Neumaier sum over its tokens in ascending order,
 *           starting from its first token: node = (sum, correction);
 *  level l>=1: nodes of level l-1 are cut into groups of 32 (the last group
 *           may be short); a group's sum is the Neumaier sum of its
 *           children's sums in ascending order (starting from the first
 *           child), with compensation c; its correction is
 *           c + (((k0 + k1) + k2) + ...), the children's corrections added in
 *           ascending order;
 *  the root is the first level with one node; the result is sum + correction.
 * The shape depends only on S.                                              */
static float tree32_column(const float *v, long stride, int S)
{
    int n = (S + TREE_FAN - 1) / TREE_FAN;
    float *sig = malloc(sizeof(float) * (size_t)n);
    float *kap = malloc(sizeof(float) * (size_t)n);
    for (int t = 0; t < n; ++t) {
        int r0 = t * TREE_FAN, r1 = r0 + TREE_FAN < S ? r0 + TREE_FAN : S;
        float s = v[(long)r0 * stride], c = 0.0f;
        for (int r = r0 + 1; r < r1; ++r) nstep_f32(&s, &c, v[(long)r * stride]);
        sig[t] = s;
        kap[t] = c;
    }
    while (n > 1) {
        int m = (n + TREE_FAN - 1) / TREE_FAN;
        for (int g = 0; g < m; ++g) {
            int i0 = g * TREE_FAN, i1 = i0 + TREE_FAN < n ? i0 + TREE_FAN : n;
            float s = sig[i0], c = 0.0f, k = kap[i0];
            for (int i = i0 + 1; i < i1; ++i) { nstep_f32(&s, &c, sig[i]); k = k + kap[i]; }
            sig[g] = s;          /* g <= i0: children already consumed */
            kap[g] = c + k;
        }
        n = m;
    }
    float res = sig[0] + kap[0];
    free(sig);
    free(kap);
    return res;
}

/* out[b,h] = the fixed 32-way tree sum over s of in[b,s,h] (S >= 1) */
void oracle_token_tree_f32(const float *in, float *out, int B, int S, int H)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            out[(size_t)b * H + h] = tree32_column(in + (size_t)b * S * H + h, H, S);
}

/* The backward's token products as the operator defines them in fp32, from
 * the forward's saved row statistics: xhat = fp32(fp32(x - mean) * rstd),
 * g = fp32(dy); prod[b,s,0:D] = fp32(g * xhat), prod[b,s,D:2D] = g.          */
void oracle_bwd_products_f32(const uint16_t *dy, const uint16_t *x, const float *mean,
                             const float *rstd, float *prod, int B, int S, int D)
{
    for (size_t row = 0; row < (size_t)B * S; ++row)
        for (int d = 0; d < D; ++d) {
            float xc = bf16_to_f32(x[row * D + d]) - mean[row];
            float xh = xc * rstd[row];
            float g = bf16_to_f32(dy[row * D + d]);
            prod[row * 2 * D + d] = g * xh;
            prod[row * 2 * D + D + d] = g;
        }
}

/* ------------------------------------------------------------------------ */
/* projection backward                                                       */
/* ------------------------------------------------------------------------ */

/* The sums of the projection backward over the output rows n0 <= n < n1:
 * d_silu[b,k] += sum_n e[b,n] W[n,k] (Neumaier accumulators acc[b*D+k]),
 * dW[n,k] = sum_b e[b,n] u[b,k], db[n] = sum_b e[b,n] (fp64, compensated).  */
static void proj_bwd_rows_core(const double *e, const double *u, const uint16_t *W, nsum *acc,
                               double *dW, double *db, int B, int D, int n0, int n1)
{
    int N = 2 * D;
    for (int b = 0; b < B; ++b)
        for (int n = n0; n < n1; ++n) {
            double en = e[(size_t)b * N + n];
            const uint16_t *w = W + (size_t)n * D;
            for (int k = 0; k < D; ++k) nsum_add(&acc[(size_t)b * D + k], en * bf16_to_f64(w[k]));
        }
    for (int n = n0; n < n1; ++n) {
        if (dW)
            for (int k = 0; k < D; ++k) {
                nsum a = {0.0, 0.0};
                for (int b = 0; b < B; ++b) nsum_add(&a, e[(size_t)b * N + n] * u[(size_t)b * D + k]);
                dW[(size_t)n * D + k] = nsum_val(&a);
            }
        if (db) {
            nsum a = {0.0, 0.0};
            for (int b = 0; b < B; ++b) nsum_add(&a, e[(size_t)b * N + n]);
            db[n] = nsum_val(&a);
        }
    }
}

/* e = bf16(d_emb); u = bf16(silu(temb));
 * d_temb[b,k] = bf16( (sum_n e[b,n] W[n,k]) * silu'(temb[b,k]) );
 * dW[n,k] = sum_b e[b,n] u[b,k];  db[n] = sum_b e[b,n]   (fp64, compensated).
 * With rows n0 <= n < n1 only (oracle_proj_bwd_rows), d_temb is replaced by
 * the fp64 partial d_silu over those rows, and dW/db cover those rows.     */
static void proj_bwd_impl(const float *d_emb, const uint16_t *temb, const uint16_t *W,
                          uint16_t *d_temb, double *d_silu, double *dW, double *db,
                          int B, int D, int n0, int n1)
{
    int N = 2 * D;
    double *e = malloc(sizeof(double) * (size_t)B * N);
    double *u = malloc(sizeof(double) * (size_t)B * D);
    nsum *acc = calloc((size_t)B * D, sizeof(nsum));
    for (size_t i = 0; i < (size_t)B * N; ++i) e[i] = bf16_to_f64(bf16_from_f32(d_emb[i]));
    for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = bf16_to_f64(bf16_from_f64(silu64(bf16_to_f64(temb[i]))));
    proj_bwd_rows_core(e, u, W, acc, dW, db, B, D, n0, n1);
    for (size_t i = 0; i < (size_t)B * D; ++i) {
        if (d_temb) d_temb[i] = bf16_from_f64(nsum_val(&acc[i]) * dsilu64(bf16_to_f64(temb[i])));
        if (d_silu) d_silu[i] = nsum_val(&acc[i]);
    }
    free(e); free(u); free(acc);
}

void oracle_proj_bwd(const float *d_emb, const uint16_t *temb, const uint16_t *W,
                     uint16_t *d_temb, double *dW, double *db, int B, int D)
{
    proj_bwd_impl(d_emb, temb, W, d_temb, NULL, dW, db, B, D, 0, 2 * D);
}

void oracle_proj_bwd_rows(const float *d_emb, const uint16_t *temb, const uint16_t *W,
                          double *d_silu, double *dW, double *db, int B, int D, int n0, int n1)
{
    proj_bwd_impl(d_emb, temb, W, NULL, d_silu, dW, db, B, D, n0, n1);
}

/* exact gradients of oracle_proj_fwd_f64 for upstream gradient d_emb */
void oracle_proj_bwd_f64(const double *d_emb, const double *temb, const double *W,
                         double *d_temb, double *dW, double *db, int B, int D)
{
    int N = 2 * D;
    for (int b = 0; b < B; ++b)
        for (int k = 0; k < D; ++k) {
            nsum a = {0.0, 0.0};
            for (int n = 0; n < N; ++n) nsum_add(&a, d_emb[(size_t)b * N + n] * W[(size_t)n * D + k]);
            d_temb[(size_t)b * D + k] = nsum_val(&a) * dsilu64(temb[(size_t)b * D + k]);
        }
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < D; ++k) {
            nsum a = {0.0, 0.0};
            for (int b = 0; b < B; ++b) nsum_add(&a, d_emb[(size_t)b * N + n] * silu64(temb[(size_t)b * D + k]));
            dW[(size_t)n * D + k] = nsum_val(&a);
        }
        nsum a = {0.0, 0.0};
        for (int b = 0; b < B; ++b) nsum_add(&a, d_emb[(size_t)b * N + n]);
        db[n] = nsum_val(&a);
    }
}

/* The weight gradient in the operator's fixed order, fp32: starting from the
 * caller's accumulators (accumulate != 0) or from +0, samples are added in
 * ascending order, acc = acc + e[b,n] * u[b,k] (the product of two bf16
 * values is exact in fp32), db_acc[n] = db_acc[n] + e[b,n].                 */
void oracle_wgrad_seq_f32(const float *d_emb, const uint16_t *temb, float *dW_acc,
                          float *db_acc, int accumulate, int B, int D)
{
    int N = 2 * D;
    float *e = malloc(sizeof(float) * (size_t)B * N);
    float *u = malloc(sizeof(float) * (size_t)B * D);
    for (size_t i = 0; i < (size_t)B * N; ++i) e[i] = bf16_to_f32(bf16_from_f32(d_emb[i]));
    for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = bf16_to_f32(bf16_from_f64(silu64(bf16_to_f64(temb[i]))));
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < D; ++k) {
            float a = accumulate ? dW_acc[(size_t)n * D + k] : 0.0f;
            for (int b = 0; b < B; ++b) a = a + e[(size_t)b * N + n] * u[(size_t)b * D + k];
            dW_acc[(size_t)n * D + k] = a;
        }
        float a = accumulate ? db_acc[n] : 0.0f;
        for (int b = 0; b < B; ++b) a = a + e[(size_t)b * N + n];
        db_acc[n] = a;
    }
    free(e); free(u);
}

/* The same order for the listed output rows only (rows[0..nrows)), each from
 * +0: dW_rows[i, k] = sum over b ascending of e[b, rows[i]] * u[b, k] in fp32,
 * db_rows[i] likewise.  For checking a sample of rows of a large batch.      */
void oracle_wgrad_seq_f32_rows(const float *d_emb, const uint16_t *temb, const int *rows, int nrows,
                               float *dW_rows, float *db_rows, int B, int D)
{
    int N = 2 * D;
    float *u = malloc(sizeof(float) * (size_t)B * D);
    for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = bf16_to_f32(bf16_from_f64(silu64(bf16_to_f64(temb[i]))));
    for (int r = 0; r < nrows; ++r) {
        int n = rows[r];
        float *dst = dW_rows + (size_t)r * D;
        for (int k = 0; k < D; ++k) dst[k] = 0.0f;
        float a = 0.0f;
        for (int b = 0; b < B; ++b) {
            float e = bf16_to_f32(bf16_from_f32(d_emb[(size_t)b * N + n]));
            for (int k = 0; k < D; ++k) dst[k] = dst[k] + e * u[(size_t)b * D + k];
            a = a + e;
        }
        db_rows[r] = a;
    }
    free(u);
}

/* ------------------------------------------------------------------------ */
/* Block-level modulated norm with a gated residual                           */
/* (ScaleResidualLayerNormScaleShift: miles_diffusion PR 108, Summary, root   */
/* cause 1 and "Patches": the norm1/norm2 sites of every block take the same  */
/* rounding points as norm_out -- fp32 LayerNorm, bf16 (1 + scale), fp32      */
/* modulation -- with the residual stream's gated add in eager bf16, each op  */
/* computed in fp32 and rounded once to bf16)                                 */
/* ------------------------------------------------------------------------ */

/* eager bf16 multiply and add: fp32 operation, one rounding to bf16 */
static uint16_t bf16_mul(uint16_t a, uint16_t b) { return bf16_from_f32(bf16_to_f32(a) * bf16_to_f32(b)); }
static uint16_t bf16_add(uint16_t a, uint16_t b) { return bf16_from_f32(bf16_to_f32(a) + bf16_to_f32(b)); }

/* r = bf16(residual + bf16(gate * x)), gate [B, D] broadcast over tokens;
 * then out, mean, rstd = LayerNorm + modulation of r (oracle_out_fwd).      */
void oracle_res_fwd(const uint16_t *x, const uint16_t *residual, const uint16_t *gate, const uint16_t *emb,
                    float eps, uint16_t *r, uint16_t *out, float *mean, float *rstd, int B, int S, int D)
{
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int d = 0; d < D; ++d) {
                size_t i = ((size_t)b * S + s) * D + d;
                r[i] = bf16_add(residual[i], bf16_mul(gate[(size_t)b * D + d], x[i]));
            }
    oracle_out_fwd(r, emb, eps, out, mean, rstd, B, S, D);
}

/* The backward's tail from the LayerNorm input's gradient dr_ln (bf16, the
 * dx of the norm_out backward applied to r) and the gradient d_r of the
 * residual output from later uses (NULL: none):
 *   gr         = bf16(dr_ln + d_r)           (autograd adds the two uses)
 *   d_residual = gr
 *   d_x        = bf16(gr * gate)
 *   d_gate     = sum_s bf16(gr * x)          (the broadcast operand's grad,
 *                                             products in eager bf16), fp32  */
void oracle_res_bwd_tail(const uint16_t *dr_ln, const uint16_t *d_r, const uint16_t *x, const uint16_t *gate,
                         uint16_t *d_x, uint16_t *d_residual, float *d_gate, int B, int S, int D)
{
    nsum *acc = malloc(sizeof(nsum) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        for (int d = 0; d < D; ++d) acc[d].s = acc[d].c = 0.0;
        for (int s = 0; s < S; ++s)
            for (int d = 0; d < D; ++d) {
                size_t i = ((size_t)b * S + s) * D + d;
                uint16_t gr = d_r ? bf16_add(dr_ln[i], d_r[i]) : dr_ln[i];
                d_residual[i] = gr;
                d_x[i] = bf16_mul(gr, gate[(size_t)b * D + d]);
                nsum_add(&acc[d], bf16_to_f64(bf16_mul(gr, x[i])));
            }
        for (int d = 0; d < D; ++d) d_gate[(size_t)b * D + d] = (float)nsum_val(&acc[d]);
    }
    free(acc);
}

/* the whole backward of oracle_res_fwd: dr_ln, d_emb from oracle_out_bwd on r */
void oracle_res_bwd(const uint16_t *d_out, const uint16_t *d_r, const uint16_t *x, const uint16_t *r,
                    const uint16_t *gate, const uint16_t *emb, float eps, uint16_t *d_x, uint16_t *d_residual,
                    float *d_emb, float *d_gate, int B, int S, int D)
{
    uint16_t *dr_ln = malloc(sizeof(uint16_t) * (size_t)B * S * D);
    oracle_out_bwd(d_out, r, emb, eps, dr_ln, d_emb, B, S, D);
    oracle_res_bwd_tail(dr_ln, d_r, x, gate, d_x, d_residual, d_gate, B, S, D);
    free(dr_ln);
}

/* the gate's token products bf16(gr * x) as fp32, the input of the fixed
 * token tree that replays d_gate (oracle_token_tree_f32)                     */
void oracle_res_gate_products_f32(const uint16_t *gr, const uint16_t *x, float *prod, long n)
{
    for (long i = 0; i < n; ++i) prod[i] = bf16_to_f32(bf16_mul(gr[i], x[i]));
}

/* ------------------------------------------------------------------------ */
/* FP32 execution dtype (RL-Kernel PR 538 "Results": the FP32 timings and the */
/* BF16/FP32 acceptance gates): the same operator on fp32 tensors with no    */
/* bf16 rounding anywhere; every eager fp32 operation rounds once to fp32.   */
/* ------------------------------------------------------------------------ */

/* u = fp32(silu(t)) (the fp32 nearest to the fp64 value);
 * emb[b,n] = fp32(sum_k u[b,k] W[n,k] + bias[n]), the sum exact (compensated
 * fp64 over the fp64-exact products of two fp32 values), rounded once.       */
void oracle_f32_proj_fwd(const float *temb, const float *W, const float *bias, float *emb, float *u, int B, int D)
{
    int N = 2 * D;
    double *ud = malloc(sizeof(double) * (size_t)B * D);
    double *wd = malloc(sizeof(double) * (size_t)N * D);
    double *bd = malloc(sizeof(double) * (size_t)N);
    double *e = malloc(sizeof(double) * (size_t)B * N);
    for (size_t i = 0; i < (size_t)B * D; ++i) {
        u[i] = (float)silu64((double)temb[i]);
        ud[i] = (double)u[i];
    }
    for (size_t i = 0; i < (size_t)N * D; ++i) wd[i] = (double)W[i];
    for (int n = 0; n < N; ++n) bd[n] = (double)bias[n];
    proj_core(ud, wd, bd, e, B, D, N, 0, N);
    for (size_t i = 0; i < (size_t)B * N; ++i) emb[i] = (float)e[i];
    free(ud); free(wd); free(bd); free(e);
}

/* xhat = fp32(exact LayerNorm of x); onep = fp32(1 + scale);
 * out = fp32(fp32(xhat * onep) + shift); mean, rstd = fp32 of the exact
 * row statistics (nullable).                                                 */
void oracle_f32_out_fwd(const float *x, const float *emb, float eps, float *out, float *mean, float *rstd, int B,
                        int S, int D)
{
    double *xr = malloc(sizeof(double) * (size_t)D);
    double *xh = malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        const float *sc = emb + (size_t)b * 2 * D, *sh = sc + D;
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            for (int d = 0; d < D; ++d) xr[d] = (double)x[row * D + d];
            double mu, r;
            ln_row(xr, D, (double)eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d) {
                float onep = 1.0f + sc[d];
                float prod = (float)xh[d] * onep;
                out[row * D + d] = prod + sh[d];
            }
            if (mean) mean[row] = (float)mu;
            if (rstd) rstd[row] = (float)r;
        }
    }
    free(xr); free(xh);
}

/* dx = fp32(exact LayerNorm backward of g * onep), g = dy, onep = fp32(1 +
 * scale); d_emb[b, 0:D] = sum_s g * fp32(xhat), d_emb[b, D:2D] = sum_s g,
 * exact sums rounded once to fp32.                                           */
void oracle_f32_out_bwd(const float *dy, const float *x, const float *emb, float eps, float *dx, float *d_emb,
                        int B, int S, int D)
{
    double *xr = malloc(sizeof(double) * (size_t)D);
    double *xh = malloc(sizeof(double) * (size_t)D);
    double *gh = malloc(sizeof(double) * (size_t)D);
    double *dxr = malloc(sizeof(double) * (size_t)D);
    nsum *ss = malloc(sizeof(nsum) * (size_t)D);
    nsum *sh = malloc(sizeof(nsum) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        const float *sc = emb + (size_t)b * 2 * D;
        for (int d = 0; d < D; ++d) ss[d].s = ss[d].c = sh[d].s = sh[d].c = 0.0;
        for (int s = 0; s < S; ++s) {
            size_t row = (size_t)b * S + s;
            for (int d = 0; d < D; ++d) xr[d] = (double)x[row * D + d];
            double mu, r;
            ln_row(xr, D, (double)eps, &mu, &r, xh);
            for (int d = 0; d < D; ++d) {
                double g = (double)dy[row * D + d];
                gh[d] = g * (double)(1.0f + sc[d]);          /* exact */
                nsum_add(&ss[d], g * (double)(float)xh[d]);  /* exact */
                nsum_add(&sh[d], g);
            }
            ln_bwd_row(gh, xh, r, D, dxr);
            for (int d = 0; d < D; ++d) dx[row * D + d] = (float)dxr[d];
        }
        for (int d = 0; d < D; ++d) {
            d_emb[(size_t)b * 2 * D + d] = (float)nsum_val(&ss[d]);
            d_emb[(size_t)b * 2 * D + D + d] = (float)nsum_val(&sh[d]);
        }
    }
    free(xr); free(xh); free(gh); free(dxr); free(ss); free(sh);
}

/* the fp32 backward's token products from saved statistics:
 * xhat = fp32(fp32(x - mean) * rstd); prod = (fp32(g * xhat), g)             */
void oracle_f32_bwd_products(const float *dy, const float *x, const float *mean, const float *rstd, float *prod,
                             int B, int S, int D)
{
    for (size_t row = 0; row < (size_t)B * S; ++row)
        for (int d = 0; d < D; ++d) {
            float xc = x[row * D + d] - mean[row];
            float xh = xc * rstd[row];
            float g = dy[row * D + d];
            prod[row * 2 * D + d] = g * xh;
            prod[row * 2 * D + D + d] = g;
        }
}

/* d_temb = fp32(sum_n e W * silu'(t)) with e = d_emb (no rounding), u =
 * fp32(silu(t)); dW = fp32(sum_b e u), db = fp32(sum_b e): exact sums,
 * rounded once (d_temb's product with silu'(t) exact in fp64 too).           */
void oracle_f32_proj_bwd(const float *d_emb, const float *temb, const float *W, float *d_temb, float *dW,
                         float *db, int B, int D)
{
    int N = 2 * D;
    nsum *acc = malloc(sizeof(nsum) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k < D; ++k) acc[k].s = acc[k].c = 0.0;
        for (int n = 0; n < N; ++n) {
            double e = (double)d_emb[(size_t)b * N + n];
            const float *w = W + (size_t)n * D;
            for (int k = 0; k < D; ++k) nsum_add(&acc[k], e * (double)w[k]);
        }
        for (int k = 0; k < D; ++k) {
            double t = (double)temb[(size_t)b * D + k];
            d_temb[(size_t)b * D + k] = (float)(nsum_val(&acc[k]) * dsilu64(t));
        }
    }
    free(acc);
    if (dW || db) {
        double *u = malloc(sizeof(double) * (size_t)B * D);
        for (size_t i = 0; i < (size_t)B * D; ++i) u[i] = (double)(float)silu64((double)temb[i]);
        for (int n = 0; n < N; ++n) {
            nsum a = {0.0, 0.0};
            if (dW)
                for (int k = 0; k < D; ++k) {
                    nsum w = {0.0, 0.0};
                    for (int b = 0; b < B; ++b) nsum_add(&w, (double)d_emb[(size_t)b * N + n] * u[(size_t)b * D + k]);
                    dW[(size_t)n * D + k] = (float)nsum_val(&w);
                }
            for (int b = 0; b < B; ++b) nsum_add(&a, (double)d_emb[(size_t)b * N + n]);
            if (db) db[n] = (float)nsum_val(&a);
        }
        free(u);
    }
}

/* The fp32 weight gradient in the operator's fixed order: from the caller's
 * accumulators (accumulate != 0) or +0, samples in ascending order, one fused
 * multiply-add per sample, acc = fma(e[b,n], u[b,k], acc) (one rounding);
 * db_acc[n] = db_acc[n] + e[b,n].  u as given (the forward's fp32 u).        */
void oracle_f32_wgrad_seq(const float *d_emb, const float *u, float *dW_acc, float *db_acc, int accumulate, int B,
                          int D)
{
    int N = 2 * D;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < D; ++k) {
            float a = accumulate ? dW_acc[(size_t)n * D + k] : 0.0f;
            for (int b = 0; b < B; ++b) a = fmaf(d_emb[(size_t)b * N + n], u[(size_t)b * D + k], a);
            dW_acc[(size_t)n * D + k] = a;
        }
        float a = accumulate ? db_acc[n] : 0.0f;
        for (int b = 0; b < B; ++b) a = a + d_emb[(size_t)b * N + n];
        db_acc[n] = a;
    }
}

/* ------------------------------------------------------------------------ */
/* proj_out: the latent projection after the final norm (RL-Kernel PR 538    */
/* "What": 3072 -> 64, latent_proj_gemm), on the bf16 output of the norm      */
/* ------------------------------------------------------------------------ */

/* y[r,j] = bf16(sum_d out[r,d] Wp[j,d] + bp[j]): the exact sum (compensated
 * fp64 over the exact products), rounded once                               */
void oracle_proj_out(const uint16_t *out, const uint16_t *Wp, const uint16_t *bp, uint16_t *y, long R, int D, int J)
{
    double *a = malloc(sizeof(double) * (size_t)D);
    double *w = malloc(sizeof(double) * (size_t)J * D);
    double *bb = malloc(sizeof(double) * (size_t)J);
    double *e = malloc(sizeof(double) * (size_t)J);
    for (size_t i = 0; i < (size_t)J * D; ++i) w[i] = bf16_to_f64(Wp[i]);
    for (int j = 0; j < J; ++j) bb[j] = bf16_to_f64(bp[j]);
    for (long r = 0; r < R; ++r) {
        for (int d = 0; d < D; ++d) a[d] = bf16_to_f64(out[(size_t)r * D + d]);
        proj_core(a, w, bb, e, 1, D, J, 0, J);
        for (int j = 0; j < J; ++j) y[(size_t)r * J + j] = bf16_from_f64(e[j]);
    }
    free(a); free(w); free(bb); free(e);
}

/* ------------------------------------------------------------------------ */
/* format helpers exported for the tests                                     */
/* ------------------------------------------------------------------------ */

void oracle_bf16_from_f64(const double *x, uint16_t *h, long n)
{
    for (long i = 0; i < n; ++i) h[i] = bf16_from_f64(x[i]);
}
