/*
 * mok_oracle.c -- plain, slow CPU oracle for one Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Pages this follows (cited by short name below):
 *   [kucoin] "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
 *            NVL72" (kucoin.com flash, Arabic), sections 01, 02, 03.
 *   [miku]   "Mixture of kittens: how Cursor opened a kernel that speeds up
 *            AI training by up to 2.4x" (miku-ai.ru news).
 * The pages give no formulas.  Each function states the plain definition it
 * computes and the reading taken where the pages are silent.
 *
 * Arithmetic is fp64 everywhere except at the layer's contract rounding
 * points (BF16 storage, MXFP8 quantisation, the fp32 fused multiply-add order
 * of the combine), which are mirrored exactly so that the GPU path can be
 * compared bit for bit where the contract says so.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC -lm
 * (-ffp-contract=off keeps a*b+c as two roundings; only the explicit fmaf of
 * the combine and reverse-dispatch contracts fuses.)
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* BF16: 8 significant bits, fp32 exponent range, round to nearest even. */
/* ------------------------------------------------------------------ */

double mko_bf16_round(double v)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    int e;
    frexp(v, &e);                       /* 2^(e-1) <= |v| < 2^e */
    int binade = e - 1;
    if (binade < -126)                  /* subnormals share the 2^-133 quantum */
        binade = -126;
    int ulp = binade - 7;
    double r = ldexp(nearbyint(ldexp(v, -ulp)), ulp);
    if (fabs(r) >= ldexp(1.0, 128))     /* rounds past the largest finite value */
        return copysign(INFINITY, v);
    return r;
}

void mko_bf16_round_array(const double *in, double *out, int64_t n)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = mko_bf16_round(in[i]);
}

/* BF16 bit pattern of a value that is already BF16-representable. */
void mko_bf16_bits_array(const double *in, uint16_t *out, int64_t n)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float f = (float)mko_bf16_round(in[i]);
        uint32_t u;
        memcpy(&u, &f, 4);
        out[i] = (uint16_t)(u >> 16);
    }
}

void mko_bf16_values_array(const uint16_t *bits, double *out, int64_t n)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)bits[i] << 16;
        float f;
        memcpy(&f, &u, 4);
        out[i] = (double)f;
    }
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 (OCP "E4M3FN"): bias 7, 3 mantissa bits, no infinities,    */
/* largest finite 448 (S.1111.110), subnormal quantum 2^-9.            */
/* Encoding is round-to-nearest-even with saturation to +-448, sign of  */
/* zero kept.                                                          */
/* ------------------------------------------------------------------ */

double mko_e4m3_decode(uint8_t c)
{
    int s = c >> 7, ef = (c >> 3) & 15, m = c & 7;
    if (ef == 15 && m == 7)
        return NAN;
    double v = (ef == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), ef - 10);
    return s ? -v : v;
}

uint8_t mko_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs(v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int binade = e - 1;
    if (binade < -6)
        binade = -6;                    /* subnormal range shares the 2^-9 quantum */
    int ulp = binade - 3;
    double r = ldexp(nearbyint(ldexp(a, -ulp)), ulp);
    if (r > 448.0)
        return (uint8_t)(sign | 0x7E);
    if (r == 0.0)
        return sign;
    frexp(r, &e);
    binade = e - 1;
    if (binade < -6)
        return (uint8_t)(sign | (uint8_t)ldexp(r, 9));
    uint8_t mant = (uint8_t)(ldexp(r, 3 - binade) - 8.0);
    return (uint8_t)(sign | (uint8_t)((binade + 7) << 3) | mant);
}

/* ------------------------------------------------------------------ */
/* MXFP8 block quantisation (OCP Microscaling Formats v1.0): one shared */
/* E8M0 scale per block of 32 consecutive elements along the GEMM's K.  */
/*   X = clamp(floor(log2(amax)) - 8, -127, 127)   (8 = E4M3 emax)       */
/*   scale byte = X + 127, element = E4M3_RNE_sat(v / 2^X)               */
/*   amax == 0 gives scale byte 0 and all elements 0.                   */
/* The pages only name MXFP8 and say activations are quantised inside  */
/* dispatch, the grouped GEMM and SwiGLU ([kucoin] §02, MXFP8 paragraph).*/
/* ------------------------------------------------------------------ */

int mko_mx_scale_exponent(double amax)
{
    if (amax == 0.0)
        return -127;
    int e;
    frexp(amax, &e);
    int x = (e - 1) - 8;
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

/* a: [rows, cols] row-major, cols % 32 == 0.  codes: [rows, cols];
 * scales: [rows, cols/32] (E8M0 bytes), blocks run along a row. */
void mko_mx_quantize(const double *a, int64_t rows, int64_t cols,
                     uint8_t *codes, uint8_t *scales)
{
    int64_t nb = cols / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double *v = a + r * cols + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs(v[i]) > amax) amax = fabs(v[i]);
            int x = mko_mx_scale_exponent(amax);
            scales[r * nb + b] = (uint8_t)(x + 127);
            for (int i = 0; i < 32; ++i)
                codes[r * cols + b * 32 + i] = mko_e4m3_encode(ldexp(v[i], -x));
        }
    }
}

void mko_mx_dequantize(const uint8_t *codes, const uint8_t *scales,
                       int64_t rows, int64_t cols, double *out)
{
    int64_t nb = cols / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = ldexp(mko_e4m3_decode(codes[r * cols + c]),
                                      (int)scales[r * nb + c / 32] - 127);
}

/* ------------------------------------------------------------------ */
/* A1 Router.  [kucoin] §01: at every step the router decides again to  */
/* which experts each token goes.  The pages give no formula; reading:  */
/*   l = x W_r^T (+ b);  s = softmax_E(l)  or  s = sigmoid(l);           */
/*   choose the k largest s, ties to the lower expert id, slot j = 0 is  */
/*   the largest;  g_j = s_j / sum over the chosen s.                    */
/* kind: 0 softmax, 1 sigmoid.                                          */
/* ------------------------------------------------------------------ */

void mko_router(int T, int d, int E, int k, int kind,
                const double *x, const double *Wr, const double *bias,
                double *logits, double *scores, int32_t *ids, double *gates)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *l = logits + (int64_t)t * E;
        double *s = scores + (int64_t)t * E;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += x[(int64_t)t * d + i] * Wr[(int64_t)e * d + i];
            l[e] = acc + (bias ? bias[e] : 0.0);
        }
        if (kind == 0) {
            double m = l[0];
            for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) z += exp(l[e] - m);
            for (int e = 0; e < E; ++e) s[e] = exp(l[e] - m) / z;
        } else {
            for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-l[e]));
        }
        double sel_sum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int q = 0; q < j; ++q) if (ids[t * k + q] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || s[e] > s[best]) best = e;   /* strict: ties keep the lower id */
            }
            ids[t * k + j] = best;
            sel_sum += s[best];
        }
        for (int j = 0; j < k; ++j)
            gates[t * k + j] = s[ids[t * k + j]] / sel_sum;
    }
}

/* ------------------------------------------------------------------ */
/* A2 Layout.  [kucoin] §01: count tokens per expert, decide where each */
/* lands on the target, keep one expert's tokens together so the        */
/* grouped GEMM gets ordered input.  Reading: a stable counting sort of  */
/* the flat slot index t*k+j by expert id.                              */
/*   counts[e], offsets = exclusive prefix sum (E+1 entries),            */
/*   slot_pos[t*k+j] = row of that slot, row_tok[p] = t, row_j[p] = j.   */
/* ------------------------------------------------------------------ */

void mko_layout(int T, int k, int E, const int32_t *ids,
                int32_t *counts, int32_t *offsets, int32_t *slot_pos,
                int32_t *row_tok, uint8_t *row_j)
{
    int64_t S = (int64_t)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < S; ++i) counts[ids[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int e = 0; e < E; ++e) {
        int32_t p = offsets[e];
        for (int64_t i = 0; i < S; ++i) {
            if (ids[i] != e) continue;
            slot_pos[i] = p;
            row_tok[p] = (int32_t)(i / k);
            row_j[p] = (uint8_t)(i % k);
            ++p;
        }
    }
}

/* ------------------------------------------------------------------ */
/* A4 SwiGLU: h = silu(a) * b, silu(a) = a / (1 + e^-a).                */
/* ------------------------------------------------------------------ */

void mko_swiglu(int64_t n, const double *a, const double *b, double *h)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        h[i] = a[i] / (1.0 + exp(-a[i])) * b[i];
}

/* ------------------------------------------------------------------ */
/* A6 Final weighted combine.  [kucoin] §03 lists the final weighted    */
/* combine as a step of the measured layer; the pages fix no order.     */
/* Contract: out[t] = bf16( fold over j = 0..k-1 of fmaf(g_tj, y_tj, acc) */
/* in fp32 starting from 0 ).  exact != 0: plain fp64 sum, no rounding. */
/* gates hold fp32 values, ystage holds BF16 values (contract mode).     */
/* ------------------------------------------------------------------ */

void mko_combine(int T, int k, int d, int exact,
                 const double *ystage, const double *gates, double *out)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            if (exact) {
                double acc = 0.0;
                for (int j = 0; j < k; ++j)
                    acc += gates[t * k + j] * ystage[((int64_t)t * k + j) * d + c];
                out[(int64_t)t * d + c] = acc;
            } else {
                float acc = 0.0f;
                for (int j = 0; j < k; ++j)
                    acc = fmaf((float)gates[t * k + j],
                               (float)ystage[((int64_t)t * k + j) * d + c], acc);
                out[(int64_t)t * d + c] = mko_bf16_round((double)acc);
            }
        }
}

/* ------------------------------------------------------------------ */
/* B1 Reverse combine ([kucoin] §02: backward pulls in reverse-combine). */
/*   dy_slot[t,j] = g_tj * dY[t]   (contract: bf16(fp32(g * dY)))        */
/*   dgates[t,j]  = < dY[t], y_tj >                                      */
/* ------------------------------------------------------------------ */

void mko_rev_combine(int T, int k, int d, int exact,
                     const double *dY, const double *gates, const double *ystage,
                     double *dy_slot, double *dgates)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            double g = gates[t * k + j];
            double dot = 0.0;
            for (int c = 0; c < d; ++c) {
                double dyv = dY[(int64_t)t * d + c];
                double v = exact ? g * dyv
                                 : mko_bf16_round((double)((float)g * (float)dyv));
                dy_slot[((int64_t)t * k + j) * d + c] = v;
                dot += dyv * ystage[((int64_t)t * k + j) * d + c];
            }
            dgates[t * k + j] = dot;
        }
}

/* ------------------------------------------------------------------ */
/* B2 SwiGLU backward: with s = sigmoid(a), silu = a s,                 */
/*   da = dh * b * s * (1 + a (1 - s)),   db = dh * silu(a).             */
/* ------------------------------------------------------------------ */

void mko_swiglu_bwd(int64_t n, const double *dh, const double *a, const double *b,
                    double *da, double *db)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double s = 1.0 / (1.0 + exp(-a[i]));
        da[i] = dh[i] * b[i] * s * (1.0 + a[i] * (1.0 - s));
        db[i] = dh[i] * a[i] * s;
    }
}

/* ------------------------------------------------------------------ */
/* B6 Router backward.  Only the chosen entries carry gradient (top-k   */
/* is piecewise constant).  With G = sum_j dg_j g_j:                      */
/*   softmax + renormalise:  dl_j = g_j (dg_j - G)                        */
/*   sigmoid + renormalise:  dl_j = (dg_j - G) / sum_sel(s) * s_j (1-s_j) */
/* dlogits [T,E] (zeros off the chosen set), dWr = dlogits^T x [E,d],    */
/* dxr = dlogits Wr [T,d].                                               */
/* ------------------------------------------------------------------ */

void mko_router_bwd(int T, int d, int E, int k, int kind,
                    const double *x, const double *Wr, const double *scores,
                    const int32_t *ids, const double *gates, const double *dgates,
                    double *dlogits, double *dWr, double *dxr)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *dl = dlogits + (int64_t)t * E;
        for (int e = 0; e < E; ++e) dl[e] = 0.0;
        double G = 0.0, sel = 0.0;
        for (int j = 0; j < k; ++j) {
            G += dgates[t * k + j] * gates[t * k + j];
            sel += scores[(int64_t)t * E + ids[t * k + j]];
        }
        for (int j = 0; j < k; ++j) {
            int e = ids[t * k + j];
            double g = gates[t * k + j], dg = dgates[t * k + j];
            if (kind == 0) {
                dl[e] = g * (dg - G);
            } else {
                double s = scores[(int64_t)t * E + e];
                dl[e] = (dg - G) / sel * s * (1.0 - s);
            }
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int e = 0; e < E; ++e)
                acc += dl[e] * Wr[(int64_t)e * d + c];
            dxr[(int64_t)t * d + c] = acc;
        }
    }
    #pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t)
                acc += dlogits[(int64_t)t * E + e] * x[(int64_t)t * d + c];
            dWr[(int64_t)e * d + c] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* B5 Reverse dispatch ([kucoin] §02: backward pushes in reverse-        */
/* dispatch) with the router's share of dX ([kucoin] §01: the router     */
/* decides at every step, so its logits carry gradient back to x):       */
/*   dX[t] = sum_j dx_slot[slot_pos[t,j]] + sum_j dl_j W_r[ids[t,j]]      */
/* where dl_j is the logit gradient of the chosen expert j (the other     */
/* logits get none).  The pages fix no order.  Contract (exact == 0):    */
/* one fp32 accumulator per element starting from 0, the k slot rows     */
/* added in ascending j, then the k router terms folded in ascending j    */
/* with fmaf(dl_j, W_r[e_j][c], acc), then BF16 round-to-nearest-even;   */
/* dx rows hold BF16 values, dl and W_r fp32 values.  exact != 0: plain   */
/* fp64 sum, no rounding.                                                 */
/* ------------------------------------------------------------------ */

void mko_rev_dispatch(int T, int k, int d, int exact,
                      const double *dx_rows, const int32_t *slot_pos,
                      const int32_t *ids, const double *dl_sel, const double *Wr,
                      double *dX)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            if (exact) {
                double acc = 0.0;
                for (int j = 0; j < k; ++j)
                    acc += dx_rows[(int64_t)slot_pos[t * k + j] * d + c];
                if (dl_sel)
                    for (int j = 0; j < k; ++j)
                        acc += dl_sel[t * k + j] * Wr[(int64_t)ids[t * k + j] * d + c];
                dX[(int64_t)t * d + c] = acc;
            } else {
                float acc = 0.0f;
                for (int j = 0; j < k; ++j)
                    acc = acc + (float)dx_rows[(int64_t)slot_pos[t * k + j] * d + c];
                if (dl_sel)
                    for (int j = 0; j < k; ++j)
                        acc = fmaf((float)dl_sel[t * k + j],
                                   (float)Wr[(int64_t)ids[t * k + j] * d + c], acc);
                dX[(int64_t)t * d + c] = mko_bf16_round((double)acc);
            }
        }
}
