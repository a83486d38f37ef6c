/*
 * ssm_oracle.c -- plain fp64 CPU definition of the selective-scan forward pass
 * (the Mamba S6 layer's scan), written to be checked by eye against the pages.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * compared with.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load or call it.  It shares no code, header,
 * table or helper with the CUDA library, and it imports nothing from it.
 *
 * What it computes (one (b, d) channel at a time, state h of N entries):
 *
 *   h[n] = h0[b,d,n], or 0 when h0 is NULL               (initial state: zeros in
 *                                                         every listing of the pages;
 *                                                         a given h0 continues a
 *                                                         sequence whose earlier part
 *                                                         ended in state h0)
 *   for t = 0 .. L-1:
 *     dt = delta[b,t,d] + (delta_bias ? delta_bias[d] : 0)
 *     if softplus_flag: dt = softplus(dt) = log(1 + exp(dt))
 *     for n:  h[n] = exp(dt * A[d,n]) * h[n] + Bbar * B[b,t,n] * u[b,t,d]
 *             Bbar = dt                                  (simplified, Euler: the default)
 *             Bbar = (exp(dt * A[d,n]) - 1) / A[d,n]     (exact zero-order hold; dt when
 *                                                         A[d,n] = 0, its limit)
 *     y      = sum_n C[b,t,n] * h[n] + (D ? D[d] : 0) * u[b,t,d]
 *     if z:   y = y * z[b,t,d] / (1 + exp(-z[b,t,d]))       (SiLU(z) gate)
 *     out[b,t,d] = y
 *   h_last[b,d,n] = h[n]
 *
 * Sources, by page and section:
 *  - "State Space Models (SSM)" summary page, section 3.2 "Selective Scan
 *    Algorithm": the pseudo-code with deltaA = exp(delta (x) A),
 *    deltaB_u = delta * B * u, x = deltaA * x + deltaB_u, y = <x, C>,
 *    x starting at zeros.  Shapes u, delta (B,L,D); A (D,N); B, C (B,L,N).
 *  - same page, section 5.1 (SelectiveSSM): dt = softplus(proj_dt(x)), where
 *    proj_dt carries a bias, so the bias is added before the softplus; the
 *    D skip term D * x.  Section 5.2 (MambaBlock): the output is multiplied by
 *    silu(z).
 *  - "Mamba와 State Space Model 논문 심층 분석" (youngju.dev), MambaBlock
 *    listing: the skip is D * x_conv, i.e. D times the scan input u, and the
 *    gate silu(z) is applied after the skip.
 *  - "상태 공간 모델" (itwiki), section "Mamba의 선택 메커니즘": the discrete
 *    transition is exp(Delta_t A), varying per token through Delta_t.
 *  - The discretisation of B is by default the simplified (Euler) form
 *    Delta * B used by every code listing on the pages.  With zoh_flag it is
 *    the exact zero-order-hold form the itwiki page prints in its "이산화"
 *    section, Bbar = (Delta A)^-1 (exp(Delta A) - I) Delta B, which for a
 *    diagonal A is (exp(Delta A_n) - 1) / A_n * B_n per state.
 *  - Obsidian "Mamba" note, section 4.2: recurrent (generation-time) inference
 *    carries only the hidden state from one token to the next, so a sequence
 *    split in two gives the same outputs when the second part starts from the
 *    first part's final state.  That is what the optional h0 means.
 *
 * Every operation is done in double precision on the exact values of the
 * inputs (the caller passes fp32 values, or bf16 values decoded exactly, as
 * doubles).  libm's exp and log1p are library primitives used as single steps.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* softplus(x) = log(1 + exp(x)), written in the overflow-free but exact form
 * max(x, 0) + log1p(exp(-|x|)).  Same value as the definition, no threshold. */
static double softplus(double x)
{
    if (x > 0.0)
        return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

/*
 * Full forward over all channels.
 *   u, delta, z : (batch, L, dim)   row-major, dim fastest
 *   A           : (dim, N)
 *   B, C        : (batch, L, N)
 *   D, delta_bias : (dim), may be NULL
 *   z           : may be NULL (no gate)
 *   h0          : (batch, dim, N) initial state, may be NULL (zeros)
 *   y           : (batch, L, dim) output
 *   h_last      : (batch, dim, N) output, may be NULL
 * Returns 0, or -1 when a required pointer is NULL, a size is negative or
 * the N-entry state cannot be allocated.
 */
int ssm_oracle_fwd_ex(const double *u, const double *delta, const double *A,
                      const double *B, const double *C, const double *D,
                      const double *z, const double *delta_bias, const double *h0,
                      int softplus_flag, int zoh_flag, double *y, double *h_last,
                      int64_t batch, int64_t L, int64_t dim, int64_t N)
{
    if (!u || !delta || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || L < 0 || dim < 0 || N < 0)
        return -1;
    double *work = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!work)
        return -1;

    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            double *h = work;
            for (int64_t n = 0; n < N; ++n)
                h[n] = h0 ? h0[(b * dim + d) * N + n] : 0.0;

            for (int64_t t = 0; t < L; ++t) {
                const int64_t i_bld = (b * L + t) * dim + d;   /* index into (B,L,D) */
                const int64_t i_bln = (b * L + t) * N;         /* row of (B,L,N)     */

                double dt = delta[i_bld];
                if (delta_bias)
                    dt += delta_bias[d];
                if (softplus_flag)
                    dt = softplus(dt);

                const double x = u[i_bld];
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double dA  = exp(dt * A[d * N + n]);       /* discretised A */
                    double dBu;
                    if (zoh_flag) {
                        const double a = A[d * N + n];
                        /* (exp(dt a) - 1) / a, and its limit dt at a = 0 */
                        const double bbar = (a != 0.0) ? expm1(dt * a) / a : dt;
                        dBu = bbar * B[i_bln + n] * x;               /* ZOH B times u */
                    } else {
                        dBu = dt * B[i_bln + n] * x;                 /* Euler B times u */
                    }
                    h[n] = dA * h[n] + dBu;
                    acc += C[i_bln + n] * h[n];
                }
                if (D)
                    acc += D[d] * x;
                if (z)
                    acc *= silu(z[i_bld]);
                y[i_bld] = acc;
            }

            if (h_last)
                for (int64_t n = 0; n < N; ++n)
                    h_last[(b * dim + d) * N + n] = h[n];
        }
    }
    free(work);
    return 0;
}

/* Euler discretisation of B, from h0. */
int ssm_oracle_fwd_h0(const double *u, const double *delta, const double *A,
                      const double *B, const double *C, const double *D,
                      const double *z, const double *delta_bias, const double *h0,
                      int softplus_flag, double *y, double *h_last,
                      int64_t batch, int64_t L, int64_t dim, int64_t N)
{
    return ssm_oracle_fwd_ex(u, delta, A, B, C, D, z, delta_bias, h0, softplus_flag, 0, y,
                             h_last, batch, L, dim, N);
}

/* The same with a zero initial state. */
int ssm_oracle_fwd(const double *u, const double *delta, const double *A,
                   const double *B, const double *C, const double *D,
                   const double *z, const double *delta_bias, int softplus_flag,
                   double *y, double *h_last,
                   int64_t batch, int64_t L, int64_t dim, int64_t N)
{
    return ssm_oracle_fwd_h0(u, delta, A, B, C, D, z, delta_bias, NULL, softplus_flag, y,
                             h_last, batch, L, dim, N);
}

/*
 * Causal depthwise 1-D convolution followed by SiLU: the step before the scan
 * in the MambaBlock listings ("Mamba와 State Space Model 논문 심층 분석",
 * youngju.dev, and the SelectiveSSM listing of the "State Space Models (SSM)"
 * summary page, section 5.1): nn.Conv1d with groups = channels, kernel size
 * K, padding K - 1 and a bias, trimmed to the first L outputs, then SiLU.
 * Conv1d is a cross-correlation over the left-padded input, so
 *
 *   u[b,t,d] = silu( sum_{k=0..K-1} w[d,k] * x[b, t - (K-1) + k, d] + cb[d] ),
 *
 * with x = 0 before t = 0 (the causal padding).
 *   x, u : (batch, L, dim)    w : (dim, K)    cb : (dim) or NULL (no bias)
 * Returns 0, or -1 for a NULL pointer or a bad size.
 */
int ssm_oracle_causal_conv_silu(const double *x, const double *w, const double *cb, double *u,
                                int64_t batch, int64_t L, int64_t dim, int64_t K)
{
    if (!x || !w || !u || batch < 0 || L < 0 || dim < 0 || K < 1)
        return -1;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t t = 0; t < L; ++t)
            for (int64_t d = 0; d < dim; ++d) {
                double acc = cb ? cb[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t s = t - (K - 1) + k;   /* input step under tap k */
                    if (s >= 0)
                        acc += w[d * K + k] * x[(b * L + s) * dim + d];
                }
                u[(b * L + t) * dim + d] = silu(acc);
            }
    return 0;
}
