/*
 * FP64 CPU oracle for the routed-expert MoE layer of the qwen3_5_moe family.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow reference that the
 * CUDA path is checked against.  Only the tests, the package's smoke check and
 * the bench's CPU-baseline leg load it; the library path never does.  It shares
 * no code, header or table with the CUDA sources.
 *
 * What it follows (page "Qwen3.6-35B-A3B (qwen3_5_moe) on the native Metal
 * engine: proposal and gate", section "What I'd build, in slices", slice
 * "The family, plain decode", and its "Gate" section):
 *   - fp32 logits over the experts and the shared expert's gate logit;
 *   - top-k by logit, ties going to the lower expert id;
 *   - pick weights exp(l - l_top) over the k picks (normalised over the picks,
 *     the "softmax top-8" of the "Qwen-3.6-35B-A3B-SIQ-K6-K4K3" model card's
 *     "Reproduction" section), rounded to bf16;
 *   - the shared expert is one more slot weighted bf16(sigmoid(bf16(gate)));
 *   - the weighted sum is rounded once to bf16;
 *   - experts are MLX affine 4-bit in groups of 64, the router 8-bit:
 *     w = scale * q + bias per group of 64 inputs of one output row;
 *   - or, the block-scaled variant: experts in NVFP4 (the checkpoint format of
 *     the page "Qwen-3.6-35B-A3B-SIQ-K6-K4K3" model card, served there by a
 *     fused FP4 MoE backend; the router stays 8-bit affine).  The pages name the
 *     format only; its definition is the public one: 4-bit E2M1 elements, one
 *     E4M3 scale per block of 16 consecutive inputs of a row, one fp32 scale
 *     per matrix, w = e2m1(q) * e4m3(s) * g.
 * The expert FFN is SwiGLU: down(silu(gate x) * up x) ("expert gate/up pair,
 * expert down" in the Gate section).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - rounding is round-to-nearest-even everywhere; fp64 goes straight to
 *     bf16 (no detour through fp32) except the logits, which the pages fix as
 *     fp32;
 *   - logit ties compare by value (+0 == -0);
 *   - the expert intermediate h stays in fp64 here;
 *   - a per-expert logit bias, when given, is added to the fp32 logit with
 *     one fp32 rounding: l = fp32(l + bias).
 *
 * Accumulation is fp64 throughout; the only roundings are the ones the
 * method names.  Tokens are independent, so every entry point works on any
 * subset of rows.  OpenMP (when compiled with -fopenmp) parallelises over
 * tokens only; each token's arithmetic is sequential and fixed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int hidden, inter, n_experts, top_k, group, bits, router_bits, has_shared;
    int format;   /* 0: MLX affine experts (bits 4 or 8), 1: NVFP4 experts */
} oracle_cfg;

#define ORACLE_NVFP4_BLOCK 16

/* ---------------------------------------------------------------- numbers */

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a finite double to the nearest bf16 (ties to even), returned as bits.
 * bf16 keeps 8 significant bits; normal exponents span [-126, 127]. */
uint16_t oracle_bf16_rne(double v)
{
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    if (isnan(v)) return 0x7FC0u;
    int neg = v < 0;
    double a = fabs(v);
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    int qe = e - 8;               /* quantum of a normal bf16 with this exponent */
    if (qe < -133) qe = -133;     /* subnormal quantum */
    double r = nearbyint(ldexp(a, -qe));   /* default mode: ties to even */
    double res = ldexp(r, qe);
    uint16_t bits;
    if (res >= 0x1p128) {
        bits = 0x7F80u;           /* overflow to infinity */
    } else {
        float f = (float)res;     /* exact: res is a bf16 value */
        uint32_t u;
        memcpy(&u, &f, 4);
        bits = (uint16_t)(u >> 16);
    }
    return (uint16_t)(bits | (neg ? 0x8000u : 0u));
}

float oracle_f32_rne(double v) { return (float)v; }

/* ---------------------------------------------------------------- dequant */

/* Dequantise one row of an affine-quantised matrix into fp64.
 * codes_row: in_dim*bits/8 bytes; for 4 bits element j sits in byte j/2,
 * low nibble for even j (MLX's uint32 packing read as little-endian bytes).
 * s_row, b_row: in_dim/group bf16 values.  w_j = s_g * q_j + b_g, g = j / group. */
void oracle_dequant_row(const uint8_t *codes_row, const uint16_t *s_row, const uint16_t *b_row,
                        int bits, int in_dim, int group, double *out)
{
    for (int j = 0; j < in_dim; ++j) {
        int q;
        if (bits == 4) {
            uint8_t byte = codes_row[j / 2];
            q = (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
        } else {
            q = codes_row[j];
        }
        int g = j / group;
        double s = oracle_bf16_to_double(s_row[g]);
        double b = oracle_bf16_to_double(b_row[g]);
        out[j] = s * (double)q + b;
    }
}

static size_t row_bytes(int in_dim, int bits) { return (size_t)in_dim * (size_t)bits / 8; }

/* E2M1, the 4-bit float of NVFP4 elements: bit 3 sign, bits 2..1 exponent
 * (bias 1), bit 0 mantissa.  Exponent 0 is subnormal: m * 2^-1.  Otherwise
 * 2^(e-1) * (1 + m/2).  No infinities, no NaN. */
double oracle_e2m1_to_double(int code)
{
    int sgn = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sgn ? -mag : mag;
}

/* E4M3 (the variant without infinities), the 8-bit float of NVFP4 block
 * scales: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * Exponent 0 is subnormal: (m/8) * 2^-6.  Otherwise 2^(e-7) * (1 + m/8).
 * Exponent 15 with mantissa 7 is NaN. */
double oracle_e4m3_to_double(int code)
{
    int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/* Dequantise one row of an NVFP4 matrix into fp64.
 * codes_row: in_dim/2 bytes, element j in byte j/2, low nibble for even j
 * (the packing of the 4-bit affine codes); s_row: in_dim/16 E4M3 bytes, one
 * per block of 16 consecutive inputs; gscale: the matrix's fp32 scale.
 * w_j = e2m1(q_j) * e4m3(s_{j/16}) * gscale, each factor exact in fp64 and
 * the product too (2 + 4 + 24 significant bits). */
void oracle_dequant_row_nvfp4(const uint8_t *codes_row, const uint8_t *s_row, float gscale, int in_dim,
                              double *out)
{
    for (int j = 0; j < in_dim; ++j) {
        uint8_t byte = codes_row[j / 2];
        int q = (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
        out[j] = oracle_e2m1_to_double(q) * oracle_e4m3_to_double(s_row[j / ORACLE_NVFP4_BLOCK]) *
                 (double)gscale;
    }
}

/* --------------------------------------------------------------- router */

/* l[t,e] = fp32( sum_h x[t,h] * w[e,h] ) with w the dequantised 8-bit router;
 * then, if bias != NULL, l = fp32(l + bias[e]). */
void oracle_router_logits(const oracle_cfg *c, const uint8_t *codes, const uint16_t *scales,
                          const uint16_t *biases, const uint16_t *x, int T, const float *bias,
                          float *logits)
{
    const int H = c->hidden, E = c->n_experts, G = c->group;
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            for (int e = 0; e < E; ++e) {
                oracle_dequant_row(codes + (size_t)e * row_bytes(H, c->router_bits),
                                   scales + (size_t)e * (H / G), biases + (size_t)e * (H / G),
                                   c->router_bits, H, G, w);
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += oracle_bf16_to_double(x[(size_t)t * H + h]) * w[h];
                float l = (float)acc;
                if (bias) l = (float)((double)l + (double)bias[e]);
                logits[(size_t)t * E + e] = l;
            }
        }
        free(w);
    }
}

/* ---------------------------------------------------------------- top-k */

/* ids[t, r] for r = 0..k-1: the r-th largest logit, ties to the lower id.
 * Plain selection: each rank scans every expert not yet taken. */
void oracle_topk(const float *logits, int T, int E, int k, int32_t *ids)
{
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int r = 0; r < k; ++r) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                /* strictly greater wins; an equal value keeps the lower id already held */
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + r] = best;
        }
    }
    free(taken);
}

/* p[t, r] = exp(l_r - l_top) / sum_j exp(l_j - l_top) over the k picks.
 * p_exact (optional) receives the fp64 value before rounding; p_bf16 the bf16 bits. */
void oracle_pick_weights(const float *logits, const int32_t *ids, int T, int E, int k,
                         double *p_exact, uint16_t *p_bf16)
{
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        const int32_t *id = ids + (size_t)t * k;
        double top = (double)l[id[0]];
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp((double)l[id[j]] - top);
        for (int j = 0; j < k; ++j) {
            double p = exp((double)l[id[j]] - top) / den;
            if (p_exact) p_exact[(size_t)t * k + j] = p;
            if (p_bf16) p_bf16[(size_t)t * k + j] = oracle_bf16_rne(p);
        }
    }
}

/* gamma[t] = fp32(sum_h x[t,h] * v[h]); w_s[t] = bf16(sigmoid(bf16(gamma))). */
void oracle_shared_weight(const uint16_t *x, const uint16_t *v, int T, int H, float *gamma,
                          uint16_t *w_s)
{
    for (int t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += oracle_bf16_to_double(x[(size_t)t * H + h]) * oracle_bf16_to_double(v[h]);
        float g = (float)acc;
        if (gamma) gamma[t] = g;
        double gb = oracle_bf16_to_double(oracle_bf16_rne((double)g));
        double sig = 1.0 / (1.0 + exp(-gb));
        if (w_s) w_s[t] = oracle_bf16_rne(sig);
    }
}

/* ---------------------------------------------------------------- expert FFN */

/* One expert matrix.  Affine: codes, scales, biases (bf16 [rows, cols/group]).
 * NVFP4: codes, bscales (E4M3 [rows, cols/16]) and gscale (fp32, one value). */
typedef struct {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *biases;
    const uint8_t *bscales;
    const float *gscale;
} oracle_qmat;

/* Pointers to expert e's block of a stacked [n, rows, cols] matrix. */
static oracle_qmat qmat_expert(const oracle_cfg *c, oracle_qmat m, int e, int rows, int cols)
{
    oracle_qmat r = m;
    if (c->format == 1) {
        r.codes = m.codes + (size_t)e * rows * row_bytes(cols, 4);
        r.bscales = m.bscales + (size_t)e * rows * (cols / ORACLE_NVFP4_BLOCK);
        r.gscale = m.gscale + e;
    } else {
        r.codes = m.codes + (size_t)e * rows * row_bytes(cols, c->bits);
        r.scales = m.scales + (size_t)e * rows * (cols / c->group);
        r.biases = m.biases + (size_t)e * rows * (cols / c->group);
    }
    return r;
}

/* y = W v for one dequantised [rows, cols] expert matrix; scratch holds cols doubles. */
static void qmat_matvec(const oracle_cfg *c, oracle_qmat m, int rows, int cols, const double *v, double *y,
                        double *scratch)
{
    const int G = c->group, bits = c->bits;
    for (int r = 0; r < rows; ++r) {
        if (c->format == 1)
            oracle_dequant_row_nvfp4(m.codes + (size_t)r * row_bytes(cols, 4),
                                     m.bscales + (size_t)r * (cols / ORACLE_NVFP4_BLOCK), *m.gscale, cols, scratch);
        else
            oracle_dequant_row(m.codes + (size_t)r * row_bytes(cols, bits), m.scales + (size_t)r * (cols / G),
                               m.biases + (size_t)r * (cols / G), bits, cols, G, scratch);
        double acc = 0.0;
        for (int j = 0; j < cols; ++j) acc += scratch[j] * v[j];
        y[r] = acc;
    }
}

/* One expert on one token, fp64 end to end:
 *   g = Wg x, u = Wu x   ([I]),  h = silu(g) * u = g / (1 + exp(-g)) * u,
 *   y = Wd h             ([H]).
 * h_out (optional) receives h.  gate/up are [I, H], down is [H, I]. */
void oracle_expert_ffn_m(const oracle_cfg *c, const oracle_qmat *mg, const oracle_qmat *mu,
                         const oracle_qmat *md, const double *x, double *h_out, double *y)
{
    const int H = c->hidden, I = c->inter;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    qmat_matvec(c, *mg, I, H, x, g, scratch);
    qmat_matvec(c, *mu, I, H, x, u, scratch);
    for (int i = 0; i < I; ++i) g[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    if (h_out) memcpy(h_out, g, sizeof(double) * (size_t)I);
    qmat_matvec(c, *md, H, I, g, y, scratch);
    free(scratch);
    free(g);
    free(u);
}

/* The same with the affine matrices given by their arrays. */
void oracle_expert_ffn(const oracle_cfg *c, const uint8_t *g_codes, const uint16_t *g_s,
                       const uint16_t *g_b, const uint8_t *u_codes, const uint16_t *u_s,
                       const uint16_t *u_b, const uint8_t *d_codes, const uint16_t *d_s,
                       const uint16_t *d_b, const double *x, double *h_out, double *y)
{
    oracle_qmat mg = {g_codes, g_s, g_b, NULL, NULL}, mu = {u_codes, u_s, u_b, NULL, NULL},
                md = {d_codes, d_s, d_b, NULL, NULL};
    oracle_expert_ffn_m(c, &mg, &mu, &md, x, h_out, y);
}

/* Down projection alone, for staged checks: y = Wd h with h given. */
void oracle_expert_down_m(const oracle_cfg *c, const oracle_qmat *md, const double *h, double *y)
{
    double *scratch = (double *)malloc(sizeof(double) * (size_t)c->inter);
    qmat_matvec(c, *md, c->hidden, c->inter, h, y, scratch);
    free(scratch);
}

void oracle_expert_down(const oracle_cfg *c, const uint8_t *d_codes, const uint16_t *d_s,
                        const uint16_t *d_b, const double *h, double *y)
{
    oracle_qmat md = {d_codes, d_s, d_b, NULL, NULL};
    oracle_expert_down_m(c, &md, h, y);
}

/* ---------------------------------------------------------------- layer */

typedef struct {
    oracle_qmat router, gate, up, down, s_gate, s_up, s_down;
    const uint16_t *shared_gate_vec;
} oracle_weights;

/* The whole layer on T tokens.
 * logits_in: [T,E] fp32 logits to use in place of the router (NULL: compute them).
 * bias: [E] fp32 per-expert logit bias (NULL: none; ignored when logits_in is given).
 * Outputs (any may be NULL except y): y bf16 [T,H]; y_exact fp64 [T,H] before the
 * final rounding; ids [T,k]; p bf16 [T,k]; w_s bf16 [T]; logits fp32 [T,E]. */
int oracle_forward(const oracle_cfg *c, const oracle_weights *w, const uint16_t *x, int T,
                   const float *bias, const float *logits_in, uint16_t *y, double *y_exact,
                   int32_t *ids_out, uint16_t *p_out, uint16_t *ws_out, float *logits_out)
{
    const int H = c->hidden, I = c->inter, E = c->n_experts, k = c->top_k;
    if (T <= 0) return 0;
    float *logits = (float *)malloc(sizeof(float) * (size_t)T * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    uint16_t *p = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * k);
    uint16_t *ws = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T);
    if (logits_in)
        memcpy(logits, logits_in, sizeof(float) * (size_t)T * E);
    else
        oracle_router_logits(c, w->router.codes, w->router.scales, w->router.biases, x, T, bias, logits);
    oracle_topk(logits, T, E, k, ids);
    oracle_pick_weights(logits, ids, T, E, k, NULL, p);
    if (c->has_shared) oracle_shared_weight(x, w->shared_gate_vec, T, H, NULL, ws);

#pragma omp parallel
    {
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        double *ye = (double *)malloc(sizeof(double) * (size_t)H);
        double *acc = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            for (int h = 0; h < H; ++h) xd[h] = oracle_bf16_to_double(x[(size_t)t * H + h]);
            for (int h = 0; h < H; ++h) acc[h] = 0.0;
            int n_slots = k + (c->has_shared ? 1 : 0);
            for (int j = 0; j < n_slots; ++j) {
                oracle_qmat mg, mu, md;
                double weight;
                if (j < k) {
                    int e = ids[(size_t)t * k + j];
                    mg = qmat_expert(c, w->gate, e, I, H);
                    mu = qmat_expert(c, w->up, e, I, H);
                    md = qmat_expert(c, w->down, e, H, I);
                    weight = oracle_bf16_to_double(p[(size_t)t * k + j]);
                } else {
                    mg = w->s_gate;
                    mu = w->s_up;
                    md = w->s_down;
                    weight = oracle_bf16_to_double(ws[t]);
                }
                oracle_expert_ffn_m(c, &mg, &mu, &md, xd, NULL, ye);
                for (int h = 0; h < H; ++h) acc[h] += weight * ye[h];
            }
            for (int h = 0; h < H; ++h) {
                if (y_exact) y_exact[(size_t)t * H + h] = acc[h];
                y[(size_t)t * H + h] = oracle_bf16_rne(acc[h]);
            }
        }
        free(xd);
        free(ye);
        free(acc);
    }
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
    if (p_out) memcpy(p_out, p, sizeof(uint16_t) * (size_t)T * k);
    if (ws_out) {
        if (c->has_shared)
            memcpy(ws_out, ws, sizeof(uint16_t) * (size_t)T);
        else
            memset(ws_out, 0, sizeof(uint16_t) * (size_t)T);
    }
    if (logits_out) memcpy(logits_out, logits, sizeof(float) * (size_t)T * E);
    free(logits);
    free(ids);
    free(p);
    free(ws);
    return 0;
}

/* ---------------------------------------------------------------- permutation */

/* Stable counting sort of the flat slots f = t*k + j by expert id.
 * counts[e] = number of slots routed to e; offsets = exclusive scan (E+1 entries);
 * perm[offsets[e] + r] = the r-th slot (in increasing f, hence increasing t) routed
 * to e; inv_perm[f] = position of f in perm. */
void oracle_permute(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv_perm)
{
    const int n = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int f = 0; f < n; ++f) counts[ids[f]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int f = 0; f < n; ++f) {
        int e = ids[f];
        int pos = offsets[e] + fill[e]++;
        perm[pos] = f;
        inv_perm[f] = pos;
    }
    free(fill);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
