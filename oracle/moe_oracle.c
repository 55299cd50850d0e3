/*
 * moe_oracle.c -- plain, slow CPU oracle for one Mixture-of-Experts layer,
 * forward and backward, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link or call this file; only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Every step is the plain definition written out as nested loops, in the
 * order the method takes them:
 *
 *   A1 router logits      L = x Wg^T (+ fixed per-expert logit bias)
 *        the gating network decides the experts of each token
 *        (ES-MoE review, section 3 "expert-wise offloading and processing"
 *         and "dynamic expert placement": placement is known only after the
 *         gating network has run)
 *   A2 softmax top-k gate.  The pages give no gate formula; this follows the
 *        plainest reading: softmax over all E logits, the k largest logits
 *        selected (lowest expert index on ties), and for k >= 2 the k
 *        probabilities renormalised to sum to one when `renorm` is set
 *   A3 per-expert histogram, exclusive prefix sum and stable assignment of
 *        tokens to their target experts, in token order
 *        (ES-MoE review, section 3: tokens are assigned to their target
 *         experts in order, with no batched matmul and no dispatch mask;
 *         FastMoE review, "proposed method": scatter/gather layout that
 *         batches the inputs by expert)
 *   A4 permute             X_perm[pos[t,j]] = x[t]
 *   A5 expert FFN forward, one expert after another over only its own
 *        contiguous segment (ES-MoE review, section 3 / section 4 table row
 *        "sequential processing"; FastMoE review: dedicated FFN with a
 *        per-expert linear, FMoETransformerMLP / FMoELinear)
 *   A6 weighted combine back to token order
 *   A7 combine backward, A8 expert FFN backward (per expert, ES-MoE review,
 *        section 3: each expert's backward pass), A9 permute backward,
 *   A10 router backward.
 *
 * Floating point: all arithmetic in double.  When `round_bf16` is non-zero
 * the activations that the bf16 configurations store in bf16 (G, A, Y_perm,
 * dY_perm, dH, dX_perm and the layer outputs y, dx) are rounded to bf16
 * (round to nearest, ties to even) at the point where they are stored; the
 * values they are computed from are never rounded.  Weight and bias
 * gradients, gate weights and logits stay in double.
 *
 * Parity pins for every function here live in tests/ (brute force, closed
 * forms, invariants, E = 1 dense FFN against a library linear layer, a dense
 * dispatch-mask formulation under torch autograd, finite differences).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---- scalar helpers ---------------------------------------------------- */

/* Round a double to the nearest bfloat16 value (8 significant bits, exponent
 * range of binary32), ties to even.  Done directly from the double so that no
 * intermediate binary32 rounding happens. */
ORACLE_API double oracle_round_bf16(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    frexp(v, &e);                 /* v = m * 2^e, 0.5 <= |m| < 1 */
    int qe = e - 8;               /* spacing of 8-significant-bit numbers */
    if (qe < -133) qe = -133;     /* bf16 subnormal spacing 2^-133 */
    double q = ldexp(1.0, qe);
    double r = nearbyint(v / q) * q;  /* default rounding mode: ties to even */
    if (fabs(r) > 3.3895313892515355e38) r = copysign(INFINITY, v);
    return r;
}

/* Elementwise oracle_round_bf16 over n values (out may alias in). */
ORACLE_API void oracle_round_bf16_array(int64_t n, const double* in, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}

static double rnd(double v, int round_bf16) {
    return round_bf16 ? oracle_round_bf16(v) : v;
}

/* GELU, exact (erf) form: x * Phi(x). */
ORACLE_API double oracle_gelu(double v) {
    return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
}

/* d/dx GELU(x) = Phi(x) + x * phi(x). */
ORACLE_API double oracle_gelu_grad(double v) {
    const double inv_sqrt_2pi = 0.3989422804014327;  /* 1/sqrt(2 pi) */
    double Phi = 0.5 * (1.0 + erf(v / sqrt(2.0)));
    double phi = inv_sqrt_2pi * exp(-0.5 * v * v);
    return Phi + v * phi;
}

/* ---- A1: router logits --------------------------------------------------- */

/* logits[t][e] = sum_c x[t][c] * Wg[e][c] + beta[e]  (beta may be NULL). */
ORACLE_API void oracle_router_logits(int64_t T, int d, int E, const double* x,
                                     const double* Wg, const double* beta,
                                     double* logits) {
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += x[t * d + c] * Wg[(int64_t)e * d + c];
            logits[t * E + e] = s + (beta ? beta[e] : 0.0);
        }
    }
}

/* ---- A2: softmax top-k gate --------------------------------------------- */

/* Softmax over all E logits of one token. */
static void softmax_row(int E, const double* L, double* p) {
    double m = L[0];
    for (int e = 1; e < E; ++e) if (L[e] > m) m = L[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(L[e] - m); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
}

/* idx[t][j]: the k experts of token t, slot j = 0 holding the largest logit;
 * equal logits go to the lower expert index.  w[t][j]: softmax probability of
 * that expert over all E experts; when renorm != 0 the k probabilities are
 * divided by their sum.  Selection compares logits, never probabilities. */
ORACLE_API void oracle_gate(int64_t T, int E, int k, int renorm,
                            const double* logits, int32_t* idx, double* w) {
    #pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * E);
        char* taken = (char*)malloc(E);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const double* L = logits + t * E;
            softmax_row(E, L, p);
            memset(taken, 0, E);
            double psum = 0.0;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    /* strictly greater: the first (lowest) index wins ties */
                    if (best < 0 || L[e] > L[best]) best = e;
                }
                taken[best] = 1;
                idx[t * k + j] = best;
                w[t * k + j] = p[best];
                psum += p[best];
            }
            if (renorm)
                for (int j = 0; j < k; ++j) w[t * k + j] /= psum;
        }
        free(p);
        free(taken);
    }
}

/* ---- A3: histogram, prefix sum, stable assignment ----------------------- */

/* counts[e] = number of (t, j) with idx[t][j] == e
 * offsets[e] = counts[0] + ... + counts[e-1], offsets[E] = T*k
 * pos[t*k+j] = offsets[e] + (number of earlier tokens t' < t routed to e)
 * perm[pos[s]] = s   (inverse permutation over the T*k slots) */
ORACLE_API void oracle_dispatch(int64_t T, int E, int k, const int32_t* idx,
                                int32_t* counts, int32_t* offsets,
                                int32_t* pos, int32_t* perm) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < T * k; ++s) counts[idx[s]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)calloc(E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t) {           /* ascending token order */
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            int32_t p = offsets[e] + cursor[e]++;
            pos[t * k + j] = p;
            perm[p] = (int32_t)(t * k + j);
        }
    }
    free(cursor);
}

/* ---- A4: permute --------------------------------------------------------- */

ORACLE_API void oracle_permute(int64_t T, int d, int k, const double* x,
                               const int32_t* pos, double* x_perm) {
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t p = pos[t * k + j];
            for (int c = 0; c < d; ++c) x_perm[p * d + c] = x[t * d + c];
        }
}

/* ---- A5: expert FFN forward ---------------------------------------------- */

/* For each expert e, one after another, over rows p in [offsets[e], offsets[e+1]):
 *   h      = W1[e] x_p + b1[e]          (W1: [E][f][d], b1: [E][f])
 *   A[p]   = GELU(h)
 *   G[p]   = GELU'(h)   (kept for the backward, which needs only this of h)
 *   Y[p]   = W2[e] A[p] + b2[e]         (W2: [E][d][f], b2: [E][d])
 * round_bf16 selects where a bf16 configuration rounds (the pages fix no
 * precision, so both plain readings are kept):
 *   1  G = GELU'(h) and A are what the forward stores, each rounded to bf16;
 *   2  the pre-activation h itself is what the forward stores (in bf16), so the
 *      backward's G = GELU'(bf16(h)), exact; A is rounded as in 1.
 * A and Y always come from the unrounded h. */
ORACLE_API void oracle_expert_ffn_fwd(int d, int f, int E, const int32_t* offsets,
                                      const double* X, const double* W1,
                                      const double* b1, const double* W2,
                                      const double* b2, double* G, double* A,
                                      double* Y, int round_bf16) {
    for (int e = 0; e < E; ++e) {
        const double* W1e = W1 + (int64_t)e * f * d;
        const double* W2e = W2 + (int64_t)e * d * f;
        #pragma omp parallel for schedule(static)
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            for (int n = 0; n < f; ++n) {
                double h = b1[(int64_t)e * f + n];
                for (int c = 0; c < d; ++c) h += W1e[(int64_t)n * d + c] * X[p * d + c];
                if (round_bf16 == 2)
                    G[p * f + n] = oracle_gelu_grad(oracle_round_bf16(h));
                else
                    G[p * f + n] = rnd(oracle_gelu_grad(h), round_bf16);
                A[p * f + n] = rnd(oracle_gelu(h), round_bf16);
            }
            for (int m = 0; m < d; ++m) {
                double y = b2[(int64_t)e * d + m];
                for (int n = 0; n < f; ++n) y += W2e[(int64_t)m * f + n] * A[p * f + n];
                Y[p * d + m] = rnd(y, round_bf16);
            }
        }
    }
}

/* ---- A6 / A9: combine (weighted un-permute) ------------------------------ */

/* y[t] = sum_j w[t][j] * Y[pos[t][j]]; with w == NULL every weight is 1, which
 * is the backward of the permute (A9). */
ORACLE_API void oracle_combine(int64_t T, int d, int k, const double* Y,
                               const int32_t* pos, const double* w, double* y,
                               int round_bf16) {
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double s = 0.0;
            for (int j = 0; j < k; ++j)
                s += (w ? w[t * k + j] : 1.0) * Y[(int64_t)pos[t * k + j] * d + c];
            y[t * d + c] = rnd(s, round_bf16);
        }
}

/* ---- A7: combine backward ------------------------------------------------ */

/* dY[pos[t][j]] = w[t][j] * dy[t];   dw[t][j] = <dy[t], Y[pos[t][j]]> */
ORACLE_API void oracle_combine_bwd(int64_t T, int d, int k, const double* dy,
                                   const double* Y, const int32_t* pos,
                                   const double* w, double* dY, double* dw,
                                   int round_bf16) {
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t p = pos[t * k + j];
            double s = 0.0;
            for (int c = 0; c < d; ++c) {
                dY[p * d + c] = rnd(w[t * k + j] * dy[t * d + c], round_bf16);
                s += dy[t * d + c] * Y[p * d + c];
            }
            dw[t * k + j] = s;
        }
}

/* ---- A8: expert FFN backward --------------------------------------------- */

/* For each expert e over its segment (chain rule through A5):
 *   dA      = W2[e]^T dY[p]
 *   dH[p]   = dA * G[p]          (G[p] = GELU'(h) from the forward)
 *   dX[p]   = W1[e]^T dH[p]
 *   dW2[e] += dY[p] A[p]^T,  db2[e] += dY[p]
 *   dW1[e] += dH[p] X[p]^T,  db1[e] += dH[p]
 * When accumulate == 0 the weight and bias gradients are overwritten. */
ORACLE_API void oracle_expert_ffn_bwd(int d, int f, int E, const int32_t* offsets,
                                      const double* dY, const double* X,
                                      const double* G, const double* A,
                                      const double* W1, const double* W2,
                                      double* dH, double* dX, double* dW1,
                                      double* db1, double* dW2, double* db2,
                                      int accumulate, int round_bf16) {
    if (!accumulate) {
        memset(dW1, 0, sizeof(double) * (size_t)E * f * d);
        memset(dW2, 0, sizeof(double) * (size_t)E * d * f);
        memset(db1, 0, sizeof(double) * (size_t)E * f);
        memset(db2, 0, sizeof(double) * (size_t)E * d);
    }
    for (int e = 0; e < E; ++e) {
        const double* W1e = W1 + (int64_t)e * f * d;
        const double* W2e = W2 + (int64_t)e * d * f;
        int64_t p0 = offsets[e], p1 = offsets[e + 1];
        /* activation gradients: rows are independent */
        #pragma omp parallel for schedule(static)
        for (int64_t p = p0; p < p1; ++p) {
            for (int n = 0; n < f; ++n) {
                double a = 0.0;
                for (int m = 0; m < d; ++m) a += W2e[(int64_t)m * f + n] * dY[p * d + m];
                dH[p * f + n] = rnd(a * G[p * f + n], round_bf16);
            }
            for (int c = 0; c < d; ++c) {
                double s = 0.0;
                for (int n = 0; n < f; ++n) s += W1e[(int64_t)n * d + c] * dH[p * f + n];
                dX[p * d + c] = rnd(s, round_bf16);
            }
        }
        /* weight gradients: sum over the expert's rows, in row order */
        #pragma omp parallel for schedule(static)
        for (int m = 0; m < d; ++m) {
            double* g = dW2 + (int64_t)e * d * f + (int64_t)m * f;
            double gb = 0.0;
            for (int64_t p = p0; p < p1; ++p) {
                double dym = dY[p * d + m];
                gb += dym;
                for (int n = 0; n < f; ++n) g[n] += dym * A[p * f + n];
            }
            db2[(int64_t)e * d + m] += gb;
        }
        #pragma omp parallel for schedule(static)
        for (int n = 0; n < f; ++n) {
            double* g = dW1 + (int64_t)e * f * d + (int64_t)n * d;
            double gb = 0.0;
            for (int64_t p = p0; p < p1; ++p) {
                double dhn = dH[p * f + n];
                gb += dhn;
                for (int c = 0; c < d; ++c) g[c] += dhn * X[p * d + c];
            }
            db1[(int64_t)e * f + n] += gb;
        }
    }
}

/* ---- A10: router backward ------------------------------------------------- */

/* Gradient of the gate weights with respect to the logits, then through A1.
 *   renorm:  w_j = softmax over the k selected logits, so
 *            dL[idx_j] = w_j (dw_j - sum_i w_i dw_i), all other dL = 0
 *   else:    w_j = p[idx_j] with p the softmax over all E logits, so
 *            dL[e] = sum_j dw_j p[idx_j] (delta(e, idx_j) - p[e])
 *   dx_r[t]  = sum_e dL[t][e] Wg[e]          (added to the permute backward)
 *   dWg[e]  += sum_t dL[t][e] x[t]   (overwritten when accumulate == 0)
 * dL (size T*E) is returned for inspection. */
ORACLE_API void oracle_router_bwd(int64_t T, int d, int E, int k, int renorm,
                                  const double* dw, const double* logits,
                                  const int32_t* idx, const double* w,
                                  const double* x, const double* Wg,
                                  double* dL, double* dx_r, double* dWg,
                                  int accumulate) {
    #pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * E);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            double* g = dL + t * E;
            for (int e = 0; e < E; ++e) g[e] = 0.0;
            if (renorm) {
                double s = 0.0;
                for (int j = 0; j < k; ++j) s += w[t * k + j] * dw[t * k + j];
                for (int j = 0; j < k; ++j)
                    g[idx[t * k + j]] = w[t * k + j] * (dw[t * k + j] - s);
            } else {
                softmax_row(E, logits + t * E, p);
                for (int j = 0; j < k; ++j) {
                    int a = idx[t * k + j];
                    for (int e = 0; e < E; ++e)
                        g[e] += dw[t * k + j] * p[a] * ((e == a ? 1.0 : 0.0) - p[e]);
                }
            }
            for (int c = 0; c < d; ++c) {
                double s = 0.0;
                for (int e = 0; e < E; ++e) s += g[e] * Wg[(int64_t)e * d + c];
                dx_r[t * d + c] = s;
            }
        }
        free(p);
    }
    if (!accumulate) memset(dWg, 0, sizeof(double) * (size_t)E * d);
    #pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t) {
            double g = dL[t * E + e];
            if (g == 0.0) continue;
            for (int c = 0; c < d; ++c) dWg[(int64_t)e * d + c] += g * x[t * d + c];
        }
}
