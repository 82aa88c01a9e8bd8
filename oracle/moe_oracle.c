/*
 * CPU oracle for the MXFP4 mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it. It shares no code, header, table or constant with the CUDA
 * library.
 *
 * It is the plain definition of the layer, written out in float64 with fixed
 * loop orders, slow on purpose:
 *   route    top-k experts per token over router logits, softmax weights
 *   permute  per-expert histogram, prefix offsets, block-padded offsets and
 *            the stable token permutation with padding rows marked -1
 *   forward  y[t] = sum_j w[t,j] * W2_e (SiLU(W1_e x_t) * (W3_e x_t)),
 *            e = ids[t,j], MXFP4 weights decoded element by element
 *
 * Sources: "DeepSeek V4 Flash 单卡 MI300X: 10 个 overlay 起家..." (txtmix.com):
 * §一 (256 experts, top-6; MoE routing then expert GEMMs), §三 (MXFP4 experts
 * with a shared E8M0 scale, the routing bitmatrix and the padding-lane mask
 * fixed to the logical block size, fused SiLU with a gate/up pair), §九 (the
 * optional SwiGLU clamp gate=min(gate,L), up=clamp(up,-L,L)). The element
 * format is the OCP Microscaling (MX) v1.0 definition of E2M1 and E8M0, which
 * the page garbles ("4-bit mantissa"): see e2m1_value below.
 *
 * Parity pins: every function here is checked against an independent
 * reference in tests/test_oracle_pins.py (format tables, brute force, closed
 * forms, library routines and a dense formulation).
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC
 * (no FMA contraction, so x86 and Arm hosts give identical results). All
 * parallel loops write disjoint outputs and keep each reduction in one
 * thread in a fixed order, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

/* E2M1 (OCP MX v1.0, FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa. Exponent field 0 is subnormal: value m * 2^-1. Otherwise
 * 2^(e-1) * (1 + m/2). All 16 codes are finite. */
double oracle_e2m1_value(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* E8M0 (OCP MX v1.0 shared scale): 2^(s-127); 0xFF is NaN. */
double oracle_e8m0_value(unsigned s)
{
    if ((s & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(s & 0xFFu) - 127);
}

/* bfloat16 bits -> exact double. */
static double bf16_value(uint16_t b)
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)b << 16;
    return (double)v.f;
}

/* Weight (row, k) of one MXFP4 matrix stored as nibbles [rows, K/2] (element
 * 2j in the low nibble of byte j) and E8M0 scales [rows, K/32]. */
static double mxfp4_weight(const uint8_t *q, const uint8_t *s, int64_t K, int64_t row, int64_t k)
{
    uint8_t byte = q[row * (K / 2) + k / 2];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 0xFu);
    return oracle_e2m1_value(code) * oracle_e8m0_value(s[row * (K / 32) + k / 32]);
}

/*
 * Routing (txtmix.com §一 / §三: each token picks top-6 of 256 experts from
 * its router scores). For each token t:
 *   ids[t, 0..k-1]  the k largest logits, in descending order; equal logits
 *                   go to the lower expert index (-0.0 equals +0.0);
 *   w[t, j]         softmax over all E logits, restricted to the chosen k and
 *                   renormalised to sum 1;
 *   bitmatrix[t,:]  optional (NULL to skip): bit e%32 of word e/32 set iff
 *                   expert e is chosen; ceil(E/32) words per token.
 * Logits must be finite.
 */
int oracle_route(const float *logits, int T, int E, int k,
                 int32_t *ids, double *w, uint32_t *bitmatrix)
{
    if (T < 0 || E < 1 || k < 1 || k > E) return ORACLE_EINVAL;
    int words = (E + 31) / 32;
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (int64_t)t * E;
        char *taken = (char *)calloc((size_t)E, 1);
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;  /* strict: lower index keeps ties */
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        /* softmax over all E, shifted by the maximum (the first chosen) */
        double lmax = (double)l[ids[(int64_t)t * k]];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - lmax); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;
        double zsel = 0.0;
        for (int j = 0; j < k; ++j) zsel += p[ids[(int64_t)t * k + j]];
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = p[ids[(int64_t)t * k + j]] / zsel;
        if (bitmatrix) {
            uint32_t *row = bitmatrix + (int64_t)t * words;
            for (int q = 0; q < words; ++q) row[q] = 0u;
            for (int j = 0; j < k; ++j) {
                int e = ids[(int64_t)t * k + j];
                row[e / 32] |= 1u << (e % 32);
            }
        }
        free(taken);
        free(p);
    }
    return ORACLE_OK;
}

/* Rows needed for the padded permutation: P + min(E, P) * (block_m - 1). */
int64_t oracle_rows_capacity(int T, int E, int k, int block_m)
{
    int64_t P = (int64_t)T * k;
    int64_t used = P < E ? P : E;
    return P + used * (block_m - 1);
}

/*
 * Permutation (txtmix.com §三: the routing bitmatrix feeds a histogram over
 * experts whose segments are padded to the kernel block size; padding lanes
 * must be masked by the logical block size, so nothing beyond the T*k real
 * (token, slot) pairs is counted). Pair p = t*k + j is token t's j-th choice.
 *   counts[e]          number of pairs routed to e
 *   offsets[0..E]      exclusive prefix sum of counts
 *   padded[0..E]       exclusive prefix sum of counts rounded up to block_m
 *   row_to_pair[r]     rows of expert e are padded[e] .. padded[e]+counts[e]-1
 *                      in ascending pair order; every other row (padding up to
 *                      padded[e+1], and the tail up to rows_capacity) is -1
 *   pair_to_row[p]     inverse map
 * Returns ORACLE_EINVAL if an id is outside [0, E).
 */
int oracle_permute(const int32_t *ids, int T, int E, int k, int block_m,
                   int32_t *counts, int32_t *offsets, int32_t *padded,
                   int32_t *row_to_pair, int64_t rows_capacity, int32_t *pair_to_row)
{
    if (T < 0 || E < 1 || k < 1 || block_m < 1) return ORACLE_EINVAL;
    int64_t P = (int64_t)T * k;
    for (int64_t p = 0; p < P; ++p)
        if (ids[p] < 0 || ids[p] >= E) return ORACLE_EINVAL;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) counts[ids[p]] += 1;
    offsets[0] = 0;
    padded[0] = 0;
    for (int e = 0; e < E; ++e) {
        offsets[e + 1] = offsets[e] + counts[e];
        int32_t c = counts[e];
        padded[e + 1] = padded[e] + (c + block_m - 1) / block_m * block_m;
    }
    if (padded[E] > rows_capacity) return ORACLE_EINVAL;
    for (int64_t r = 0; r < rows_capacity; ++r) row_to_pair[r] = -1;
    for (int e = 0; e < E; ++e) {
        int32_t next = padded[e];
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) {
                row_to_pair[next] = (int32_t)p;
                pair_to_row[p] = next;
                ++next;
            }
    }
    return ORACLE_OK;
}

/* SiLU(g) = g / (1 + exp(-g)), written to stay finite for large |g|. */
static double silu(double g)
{
    return g >= 0.0 ? g / (1.0 + exp(-g)) : g * exp(g) / (1.0 + exp(g));
}

/*
 * Layer output for the tokens listed in tok[0..n_tok-1] (txtmix.com §三:
 * grouped MXFP4 expert GEMMs with SiLU fused on the gate/up pair; §九: the
 * optional clamp). For token t and slot j with expert e = ids[t,j]:
 *   g[n] = sum_h x[t,h] * W13[e][n][h],      n in [0, I)      (gate, W1)
 *   u[n] = sum_h x[t,h] * W13[e][I+n][h]                      (up, W3)
 *   if swiglu_limit > 0: g = min(g, L), u = clamp(u, -L, L)
 *   a[n] = SiLU(g[n]) * u[n]
 *   o[c] = sum_n a[n] * W2[e][c][n],         c in [0, H)
 *   y[i, c] = sum_j w[t,j] * o_j[c]          (j ascending)
 * Weights are decoded element by element; everything is float64. y is
 * [n_tok, H], row i for token tok[i].
 */
int oracle_forward(const uint16_t *x_bf16,
                   const uint8_t *w13_q, const uint8_t *w13_s,
                   const uint8_t *w2_q, const uint8_t *w2_s,
                   const int32_t *ids, const double *w,
                   int T, int H, int I, int E, int k, double swiglu_limit,
                   const int32_t *tok, int n_tok, double *y)
{
    if (T < 0 || H < 32 || I < 32 || H % 32 || I % 32 || E < 1 || k < 1 || n_tok < 0)
        return ORACLE_EINVAL;
    for (int i = 0; i < n_tok; ++i) {
        if (tok[i] < 0 || tok[i] >= T) return ORACLE_EINVAL;
        for (int j = 0; j < k; ++j) {
            int32_t e = ids[(int64_t)tok[i] * k + j];
            if (e < 0 || e >= E) return ORACLE_EINVAL;
        }
    }
    const int64_t K13 = H, K2 = I;
    const int64_t rows13 = 2 * (int64_t)I, rows2 = H;
    int64_t nslot = (int64_t)n_tok * k;
    double *act = (double *)malloc(sizeof(double) * (size_t)(nslot * I + 1));
    double *out = (double *)malloc(sizeof(double) * (size_t)(nslot * H + 1));

    /* a = SiLU(W1 x) * (W3 x) for every (token, slot, n) */
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t idx = 0; idx < nslot * I; ++idx) {
        int64_t sl = idx / I, n = idx % I;
        int t = tok[sl / k];
        int32_t e = ids[(int64_t)t * k + sl % k];
        const uint8_t *q = w13_q + (int64_t)e * rows13 * (K13 / 2);
        const uint8_t *s = w13_s + (int64_t)e * rows13 * (K13 / 32);
        const uint16_t *xt = x_bf16 + (int64_t)t * H;
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < K13; ++h) {
            double xv = bf16_value(xt[h]);
            g += xv * mxfp4_weight(q, s, K13, n, h);
            u += xv * mxfp4_weight(q, s, K13, I + n, h);
        }
        if (swiglu_limit > 0.0) {
            if (g > swiglu_limit) g = swiglu_limit;
            if (u > swiglu_limit) u = swiglu_limit;
            if (u < -swiglu_limit) u = -swiglu_limit;
        }
        act[idx] = silu(g) * u;
    }

    /* o = W2 a for every (token, slot, c) */
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t idx = 0; idx < nslot * H; ++idx) {
        int64_t sl = idx / H, c = idx % H;
        int t = tok[sl / k];
        int32_t e = ids[(int64_t)t * k + sl % k];
        const uint8_t *q = w2_q + (int64_t)e * rows2 * (K2 / 2);
        const uint8_t *s = w2_s + (int64_t)e * rows2 * (K2 / 32);
        const double *a = act + sl * I;
        double acc = 0.0;
        for (int64_t n = 0; n < K2; ++n) acc += a[n] * mxfp4_weight(q, s, K2, c, n);
        out[idx] = acc;
    }

    /* y = sum_j w[t,j] * o_j, slots in ascending order */
    #pragma omp parallel for schedule(static)
    for (int64_t idx = 0; idx < (int64_t)n_tok * H; ++idx) {
        int64_t i = idx / H, c = idx % H;
        int t = tok[i];
        double acc = 0.0;
        for (int j = 0; j < k; ++j) acc += w[(int64_t)t * k + j] * out[(i * k + j) * H + c];
        y[idx] = acc;
    }
    free(act);
    free(out);
    return ORACLE_OK;
}

/*
 * The same layer in its grouped (permuted) form: rows of the padded
 * permutation are processed expert segment by expert segment, padding rows
 * (row_to_pair == -1) carry a zero activation row, and the weighted outputs
 * are scattered back to token order. It exists to check, inside the oracle,
 * that the permutation and padding of oracle_permute reproduce the plain
 * definition (padding rows contribute zero). y is [T, H].
 */
int oracle_forward_grouped(const uint16_t *x_bf16,
                           const uint8_t *w13_q, const uint8_t *w13_s,
                           const uint8_t *w2_q, const uint8_t *w2_s,
                           const double *w, const int32_t *padded, const int32_t *row_to_pair,
                           int T, int H, int I, int E, int k, double swiglu_limit, double *y)
{
    if (T < 0 || H % 32 || I % 32 || E < 1 || k < 1) return ORACLE_EINVAL;
    const int64_t K13 = H, K2 = I;
    int64_t R = padded[E];
    double *o = (double *)calloc((size_t)(R * H + 1), sizeof(double));
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        int e = 0;
        while (!(padded[e] <= r && r < padded[e + 1])) ++e;
        int32_t p = row_to_pair[r];
        double *xr = (double *)calloc((size_t)H, sizeof(double));
        double *a = (double *)malloc(sizeof(double) * (size_t)I);
        if (p >= 0)
            for (int64_t h = 0; h < H; ++h) xr[h] = bf16_value(x_bf16[(int64_t)(p / k) * H + h]);
        const uint8_t *q13 = w13_q + (int64_t)e * 2 * I * (K13 / 2);
        const uint8_t *s13 = w13_s + (int64_t)e * 2 * I * (K13 / 32);
        for (int64_t n = 0; n < I; ++n) {
            double g = 0.0, u = 0.0;
            for (int64_t h = 0; h < K13; ++h) {
                g += xr[h] * mxfp4_weight(q13, s13, K13, n, h);
                u += xr[h] * mxfp4_weight(q13, s13, K13, I + n, h);
            }
            if (swiglu_limit > 0.0) {
                if (g > swiglu_limit) g = swiglu_limit;
                if (u > swiglu_limit) u = swiglu_limit;
                if (u < -swiglu_limit) u = -swiglu_limit;
            }
            a[n] = silu(g) * u;
        }
        const uint8_t *q2 = w2_q + (int64_t)e * H * (K2 / 2);
        const uint8_t *s2 = w2_s + (int64_t)e * H * (K2 / 32);
        for (int64_t c = 0; c < H; ++c) {
            double acc = 0.0;
            for (int64_t n = 0; n < K2; ++n) acc += a[n] * mxfp4_weight(q2, s2, K2, c, n);
            o[r * H + c] = acc;
        }
        free(xr);
        free(a);
    }
    /* scatter-combine: token t gathers its k rows in slot order */
    for (int64_t i = 0; i < (int64_t)T * H; ++i) y[i] = 0.0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t p = (int64_t)t * k + j;
            int64_t r = -1;
            for (int64_t rr = 0; rr < R; ++rr) if (row_to_pair[rr] == p) { r = rr; break; }
            if (r < 0) { free(o); return ORACLE_EINVAL; }
            for (int64_t c = 0; c < H; ++c) y[(int64_t)t * H + c] += w[p] * o[r * H + c];
        }
    free(o);
    return ORACLE_OK;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
