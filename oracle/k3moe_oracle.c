/*
 * k3moe_oracle.c -- plain fp64 CPU definition of the Kimi K3 latent routed-MoE
 * layer forward.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.  It
 * shares no code, header or table with the CUDA library.
 *
 * Every step is the plain definition, in the order the sources give it, with
 * every intermediate kept in fp64 and no blocking or fusion:
 *
 *   1. MXFP4 weights.  "Kimi K3, as released", section "Gate 3 repeated on real
 *      K3 experts": weight_packed holds two E2M1 codes per byte, low nibble
 *      first; weight_scale holds one E8M0 exponent per 32 weights whose value is
 *      exactly 2^(e-127).  The E2M1 code is decoded from its bits as the OCP
 *      Microscaling v1.0 element format defines it (1 sign bit, 2 exponent bits
 *      with bias 1, 1 mantissa bit, exponent 0 subnormal); the GGUF notes
 *      ("quants.md", MXFP4 row) name the element type "4-bit E2M1".
 *   2. Router.  "Kimi K3, as released", table "Shape" (router: sigmoid, 1 group,
 *      routed_scaling_factor 1.0) and section "Against the technical report"
 *      (e_score_correction_bias for selection only, weights renormalized over
 *      the selected top-k, then routed_scaling_factor).  logits l = x W_r^T,
 *      scores s = sigmoid(l); the selection key is l (no bias; sigmoid is
 *      strictly increasing, so this orders exactly like s) or s + b (bias);
 *      top-K by key, descending, exact ties to the lower expert index.
 *      w_k = s_k / sum_sel s * routed_scaling_factor (bias never enters w).
 *   3. Latent MoE.  "Kimi K3, as released", section "The headline correction"
 *      and the review's "Stable LatentMoE" section (routed path: down
 *      projection -> gated experts -> aggregation -> normalisation -> up
 *      projection): h = W_down x; per selected expert y_e = W2 (act(W1 h) * W3 h)
 *      with act = SiLU (w1 = gate, w3 = up), or the SiTU reading below;
 *      z = sum_k w_k y_k;
 *      n = z / sqrt(mean(z^2) + eps) * gamma (routed_expert_norm, RMSNorm before
 *      the up-projection); o = W_up n.
 *   4. Shared experts (optional).  The review's parameter section: two shared
 *      experts always on, on the full 7168 hidden, merged into one GLU of width
 *      2 x 3072 = 6144; o += W2s (act(W1s x) * W3s x).
 *
 *   5. SiTU-GLU (optional activation).  "Kimi K3, as released", section "What
 *      is new since Kimi-Linear", item 3 (hidden_act "situ", Sigmoid Tanh Unit,
 *      activation_situ_beta 4, activation_situ_linear_beta 25) and the review's
 *      "SiTU-GLU is a soft fuse" section (sigmoid and tanh soft limits on the
 *      two GLU branches; each output coordinate bounded by 100; near the origin
 *      beta tanh(z/beta) = z + O(z^3/beta^2), so the unit is locally SwiGLU).
 *      The pages print no formula.  Reading: SiLU's linear factor g is
 *      soft-limited, and so is the linear (up) branch:
 *        act(g, u) = sigmoid(g) * beta tanh(g/beta) * linear_beta tanh(u/linear_beta).
 *      Parity unpinned beyond the bound and the two limits the pages state.
 *   6. A8 (optional).  The review's post-training section: from SFT on, the
 *      routed experts were trained with MXFP4 weights and MXFP8 input
 *      activations; attention, the latent projections, the shared experts and
 *      the router keep higher precision.  So the two activation inputs of the
 *      routed expert GEMMs -- h, and the GLU output a -- are quantised to MXFP8
 *      per token along the reduction axis: OCP Microscaling v1.0 E4M3 elements
 *      (round to nearest even, saturating at +-448) with one E8M0 scale per 32,
 *      X = floor(log2 amax) - 8.  Reading: h is quantised from its BF16 value
 *      (the precision the layer stores it in), a from its unrounded value.
 *
 * Precision: inputs widen exactly (BF16/fp32 -> fp64); all arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------ formats */

/* BF16 bit pattern -> fp64 (exact). */
double oracle_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E2M1 code (4 bits) -> value, from the bit fields of the OCP MX element format. */
double oracle_e2m1(unsigned code)
{
    unsigned sign = (code >> 3) & 1u;
    unsigned expo = (code >> 1) & 3u;
    unsigned mant = code & 1u;
    double mag;
    if (expo == 0)
        mag = 0.5 * (double)mant;                                /* subnormal: 0.m x 2^(1-1) */
    else
        mag = ldexp(1.0 + 0.5 * (double)mant, (int)expo - 1);   /* 1.m x 2^(e-1) */
    return sign ? -mag : mag;
}

/* E8M0 exponent byte -> 2^(e-127).  255 (NaN) is rejected by the caller. */
double oracle_e8m0(unsigned e)
{
    return ldexp(1.0, (int)e - 127);
}

/* fp64 -> nearest BF16 value (ties to even), as fp64. */
double oracle_round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    int e;
    double m = frexp(v, &e);                     /* v = m 2^e, 0.5 <= |m| < 1 */
    return ldexp(nearbyint(ldexp(m, 8)), e - 8); /* 8 significant bits */
}

/* fp64 -> nearest OCP E4M3 value (bias 7, 3 mantissa bits, subnormal spacing
 * 2^-9, ties to even), saturating at +-448. */
double oracle_e4m3(double v)
{
    double a = fabs(v);
    if (a == 0.0 || isnan(v))
        return v;
    int e;
    frexp(a, &e);                                /* a = m 2^e, 0.5 <= m < 1: floor(log2 a) = e - 1, exactly */
    e -= 1;
    if (e < -6)
        e = -6;                                  /* subnormals: spacing stays 2^-9 */
    double step = ldexp(1.0, e - 3);
    double q = nearbyint(a / step) * step;
    if (q > 448.0)
        q = 448.0;
    return v < 0 ? -q : q;
}

/* One row of n values (n a multiple of 32) -> MXFP8 values: per block of 32,
 * X = floor(log2 amax) - 8 (kept in [-127, 127]) and E4M3(v / 2^X) 2^X. */
void oracle_mxfp8_row(const double *in, int n, double *out)
{
    for (int b = 0; b < n / 32; b++) {
        double amax = 0.0;
        for (int j = 0; j < 32; j++)
            amax = fmax(amax, fabs(in[32 * b + j]));
        if (amax == 0.0) {
            for (int j = 0; j < 32; j++)
                out[32 * b + j] = 0.0;
            continue;
        }
        int X;
        frexp(amax, &X);                         /* floor(log2 amax) = X - 1, exact (no log2 rounding) */
        X -= 1 + 8;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
        for (int j = 0; j < 32; j++)
            out[32 * b + j] = ldexp(oracle_e4m3(ldexp(in[32 * b + j], -X)), X);
    }
}

/* Dequantise one row of n MXFP4 values (n a multiple of 32). */
void oracle_dequant_row(const uint8_t *packed, const uint8_t *scale, int n, double *out)
{
    double table[16];
    for (unsigned c = 0; c < 16; c++)
        table[c] = oracle_e2m1(c);
    for (int b = 0; b < n / 32; b++) {
        double s = oracle_e8m0(scale[b]);
        for (int j = 0; j < 32; j++) {
            int k = 32 * b + j;
            uint8_t byte = packed[k / 2];
            unsigned code = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);  /* low nibble first */
            out[k] = table[code] * s;
        }
    }
}

/* ------------------------------------------------------------ inputs */

typedef struct {
    int H, L, E, K, I, S;        /* hidden, latent, experts, top-k, expert inter, shared inter (0 = none) */
    double rms_eps, routed_scaling;
    int router_bf16;             /* 1: W_router holds BF16 bits; 0: fp32 */
    int has_bias;
    int act;                     /* 0: SiLU; 1: SiTU */
    double situ_beta, situ_linear_beta;
    int a8;                      /* 1: MXFP8 activations into the routed experts (step 6) */
} oracle_cfg;

typedef struct {
    const void *w_router;        /* [E, H] fp32 or BF16 bits */
    const float *bias;           /* [E] or NULL */
    const uint16_t *w_down;      /* [L, H] BF16 */
    const uint16_t *w_up;        /* [H, L] BF16 */
    const uint16_t *gamma;       /* [L] BF16 */
    /* per expert (NULL allowed for experts no requested token selects) */
    const uint8_t *const *w1p, *const *w1s, *const *w3p, *const *w3s, *const *w2p, *const *w2s;
    /* shared GLU (used when S > 0) */
    const uint8_t *ws1p, *ws1s, *ws3p, *ws3s, *ws2p, *ws2s;
} oracle_weights;

static double router_weight(const oracle_cfg *c, const oracle_weights *w, int j, int k)
{
    size_t i = (size_t)j * c->H + k;
    if (c->router_bf16)
        return oracle_bf16(((const uint16_t *)w->w_router)[i]);
    return (double)((const float *)w->w_router)[i];
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }
static double silu(double v) { return v * sigmoid(v); }

/* The GLU activation of gate g and up u (step 3; step 5 for SiTU). */
double oracle_act(int act, double beta, double linear_beta, double g, double u)
{
    if (act == 1) return sigmoid(g) * beta * tanh(g / beta) * linear_beta * tanh(u / linear_beta);
    return silu(g) * u;
}

/* ------------------------------------------------------------ router */

/*
 * Route one token.  Outputs idx[K], wts[K] (selection order: key descending,
 * ties to the lower index), the key gap between the K-th and (K+1)-th keys
 * (+inf when K == E), and optionally logits[E].
 */
static void route_token(const oracle_cfg *c, const oracle_weights *w, const uint16_t *xrow,
                        int *idx, double *wts, double *gap, double *logits_out)
{
    int E = c->E, K = c->K;
    double *l = (double *)malloc(sizeof(double) * E);
    double *key = (double *)malloc(sizeof(double) * E);
    char *taken = (char *)calloc(E, 1);
    for (int j = 0; j < E; j++) {
        double acc = 0.0;
        for (int k = 0; k < c->H; k++)
            acc += oracle_bf16(xrow[k]) * router_weight(c, w, j, k);
        l[j] = acc;
        key[j] = c->has_bias ? sigmoid(acc) + (double)w->bias[j] : acc;
        if (logits_out)
            logits_out[j] = acc;
    }
    double ssum = 0.0;
    for (int s = 0; s < K; s++) {
        int best = -1;
        for (int j = 0; j < E; j++) {
            if (taken[j])
                continue;
            if (best < 0 || key[j] > key[best])   /* strict '>' keeps the lower index on ties */
                best = j;
        }
        taken[best] = 1;
        idx[s] = best;
        ssum += sigmoid(l[best]);
    }
    double next = -INFINITY;
    int have_next = 0;
    for (int j = 0; j < E; j++)
        if (!taken[j] && (!have_next || key[j] > next)) {
            next = key[j];
            have_next = 1;
        }
    *gap = have_next ? key[idx[K - 1]] - next : INFINITY;
    for (int s = 0; s < K; s++)
        wts[s] = sigmoid(l[idx[s]]) / ssum * c->routed_scaling;
    free(l);
    free(key);
    free(taken);
}

/* Route n tokens (rows of x given by tokens[]); parallel over tokens. */
void oracle_route(const oracle_cfg *c, const oracle_weights *w, const uint16_t *x,
                  const int64_t *tokens, int n, int *idx, double *wts, double *gap,
                  double *logits, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int i = 0; i < n; i++)
        route_token(c, w, x + (size_t)tokens[i] * c->H, idx + (size_t)i * c->K,
                    wts + (size_t)i * c->K, gap + i, logits ? logits + (size_t)i * c->E : NULL);
}

/* ------------------------------------------------------------ GLU expert */

/*
 * out[t] += coef[t] * W2 (act(W1 in[t]) * W3 in[t]) for t < ntok, with the three
 * MXFP4 matrices dequantised row by row.  in: [ntok][din], out: [ntok][dout].
 */
static void glu_apply(const oracle_cfg *c, const uint8_t *w1p, const uint8_t *w1s, const uint8_t *w3p,
                      const uint8_t *w3s, const uint8_t *w2p, const uint8_t *w2s, int din, int dint, int dout,
                      int ntok, const double *in, const double *coef, double *out, int q8)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)ntok * dint);
    /* gate/up projections and activation */
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *r1 = (double *)malloc(sizeof(double) * din);
        double *r3 = (double *)malloc(sizeof(double) * din);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int r = 0; r < dint; r++) {
            oracle_dequant_row(w1p + (size_t)r * (din / 2), w1s + (size_t)r * (din / 32), din, r1);
            oracle_dequant_row(w3p + (size_t)r * (din / 2), w3s + (size_t)r * (din / 32), din, r3);
            for (int t = 0; t < ntok; t++) {
                const double *v = in + (size_t)t * din;
                double g = 0.0, u = 0.0;
                for (int k = 0; k < din; k++) {
                    g += r1[k] * v[k];
                    u += r3[k] * v[k];
                }
                a[(size_t)t * dint + r] = oracle_act(c->act, c->situ_beta, c->situ_linear_beta, g, u);
            }
        }
        free(r1);
        free(r3);
    }
    /* step 6: the down projection's input in MXFP8 */
    if (q8)
        for (int t = 0; t < ntok; t++)
            oracle_mxfp8_row(a + (size_t)t * dint, dint, a + (size_t)t * dint);
    /* down projection */
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *r2 = (double *)malloc(sizeof(double) * dint);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int r = 0; r < dout; r++) {
            oracle_dequant_row(w2p + (size_t)r * (dint / 2), w2s + (size_t)r * (dint / 32), dint, r2);
            for (int t = 0; t < ntok; t++) {
                const double *v = a + (size_t)t * dint;
                double y = 0.0;
                for (int k = 0; k < dint; k++)
                    y += r2[k] * v[k];
                out[(size_t)t * dout + r] += coef[t] * y;
            }
        }
        free(r2);
    }
    free(a);
}

/* ------------------------------------------------------------ forward */

/*
 * Full forward for n tokens (rows tokens[] of x).  Outputs:
 *   out [n, H] fp64, idx [n, K], wts [n, K], gap [n];
 *   h_out [n, L] (optional, the latent), z_out [n, L] (optional, the combine).
 * Returns 0, or -1 when a selected expert has NULL weights, -2 on a 255 scale.
 */
int oracle_forward(const oracle_cfg *c, const oracle_weights *w, const uint16_t *x,
                   const int64_t *tokens, int n, double *out, int *idx, double *wts, double *gap,
                   double *h_out, double *z_out, int nthreads)
{
    int H = c->H, L = c->L, E = c->E, K = c->K;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#endif
    /* 2. routing */
    oracle_route(c, w, x, tokens, n, idx, wts, gap, NULL, nthreads);

    /* 3a. latent h = W_down x */
    double *xin = (double *)malloc(sizeof(double) * (size_t)n * H);
    double *h = (double *)malloc(sizeof(double) * (size_t)n * L);
    for (int i = 0; i < n; i++)
        for (int k = 0; k < H; k++)
            xin[(size_t)i * H + k] = oracle_bf16(x[(size_t)tokens[i] * H + k]);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int r = 0; r < L; r++)
        for (int i = 0; i < n; i++) {
            double acc = 0.0;
            for (int k = 0; k < H; k++)
                acc += oracle_bf16(w->w_down[(size_t)r * H + k]) * xin[(size_t)i * H + k];
            h[(size_t)i * L + r] = acc;
        }
    /* step 6: the routed experts' input h, stored BF16, in MXFP8 */
    if (c->a8)
        for (int i = 0; i < n; i++) {
            double *hr = h + (size_t)i * L;
            for (int r = 0; r < L; r++)
                hr[r] = oracle_round_bf16(hr[r]);
            oracle_mxfp8_row(hr, L, hr);
        }

    /* 3b. experts, expert by expert in index order; z accumulates w_k y_k */
    double *z = (double *)calloc((size_t)n * L, sizeof(double));
    int rc = 0;
    int *members = (int *)malloc(sizeof(int) * (size_t)n * K);
    double *in = (double *)malloc(sizeof(double) * (size_t)n * K * L);
    double *coef = (double *)malloc(sizeof(double) * (size_t)n * K);
    double *y = (double *)malloc(sizeof(double) * (size_t)n * K * L);
    for (int e = 0; e < E && rc == 0; e++) {
        int m = 0;
        for (int i = 0; i < n; i++)
            for (int s = 0; s < K; s++)
                if (idx[(size_t)i * K + s] == e) {
                    members[m] = i;
                    coef[m] = wts[(size_t)i * K + s];
                    memcpy(in + (size_t)m * L, h + (size_t)i * L, sizeof(double) * L);
                    m++;
                }
        if (m == 0)
            continue;
        if (!w->w1p[e] || !w->w1s[e] || !w->w3p[e] || !w->w3s[e] || !w->w2p[e] || !w->w2s[e]) {
            rc = -1;
            break;
        }
        const uint8_t *sc[3] = {w->w1s[e], w->w3s[e], w->w2s[e]};
        size_t nsc[3] = {(size_t)c->I * (L / 32), (size_t)c->I * (L / 32), (size_t)L * (c->I / 32)};
        for (int q = 0; q < 3; q++)
            for (size_t j = 0; j < nsc[q]; j++)
                if (sc[q][j] == 255)
                    rc = -2;
        if (rc)
            break;
        memset(y, 0, sizeof(double) * (size_t)m * L);
        glu_apply(c, w->w1p[e], w->w1s[e], w->w3p[e], w->w3s[e], w->w2p[e], w->w2s[e],
                  L, c->I, L, m, in, coef, y, c->a8);
        for (int q = 0; q < m; q++)
            for (int r = 0; r < L; r++)
                z[(size_t)members[q] * L + r] += y[(size_t)q * L + r];
    }

    /* 3c. RMSNorm and up-projection */
    double *nrm = (double *)malloc(sizeof(double) * (size_t)n * L);
    for (int i = 0; i < n && rc == 0; i++) {
        double ms = 0.0;
        for (int r = 0; r < L; r++)
            ms += z[(size_t)i * L + r] * z[(size_t)i * L + r];
        ms /= (double)L;
        double inv = 1.0 / sqrt(ms + c->rms_eps);
        for (int r = 0; r < L; r++)
            nrm[(size_t)i * L + r] = z[(size_t)i * L + r] * inv * oracle_bf16(w->gamma[r]);
    }
    if (rc == 0) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int r = 0; r < H; r++)
            for (int i = 0; i < n; i++) {
                double acc = 0.0;
                for (int k = 0; k < L; k++)
                    acc += oracle_bf16(w->w_up[(size_t)r * L + k]) * nrm[(size_t)i * L + k];
                out[(size_t)i * H + r] = acc;
            }
    }

    /* 4. shared experts on the full hidden state, summed into the output */
    if (rc == 0 && c->S > 0) {
        double *ones = (double *)malloc(sizeof(double) * n);
        for (int i = 0; i < n; i++)
            ones[i] = 1.0;
        glu_apply(c, w->ws1p, w->ws1s, w->ws3p, w->ws3s, w->ws2p, w->ws2s, H, c->S, H, n, xin, ones, out, 0);
        free(ones);
    }

    if (rc == 0 && h_out)
        memcpy(h_out, h, sizeof(double) * (size_t)n * L);
    if (rc == 0 && z_out)
        memcpy(z_out, z, sizeof(double) * (size_t)n * L);
    free(xin);
    free(h);
    free(z);
    free(members);
    free(in);
    free(coef);
    free(y);
    free(nrm);
    return rc;
}

/* Number of threads OpenMP will use (for reporting the CPU-baseline core count). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
