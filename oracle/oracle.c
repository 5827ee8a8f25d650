/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the selective state-space
 * scan, its scalar-A-per-head chunked SSD form and its single-token decode
 * step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library; the two meet only through seeded inputs.
 *
 * Every quantity is computed in double precision, in the order the pages
 * state it, one time step after another.  Loops over independent rows
 * (batch x channel, batch x head x headdim) are spread over OpenMP threads;
 * nothing inside a row is reordered.
 *
 * Sources (page title, section):
 *  [P1] "We brought Mamba to Trainium -- and mapped where custom kernels
 *       actually help", section "Mamba: bringing an unsupported model to the
 *       chip, and writing its missing kernel": the recurrence
 *       h_t = A_t h_{t-1} + B_t x_t and the read-out y_t = sum_n C_t h_t.
 *  [P1] same page, section "We built the parallel scan -- and it taught us
 *       something sharper": the recurrence is associative, so it may be
 *       evaluated as a combination of pieces (used by oracle_scan_pieces).
 *  [P2] "Mamba-3 NKI Kernels for AWS Neuron", section "How it works",
 *       Phase 0: dt = softplus(dt + dt_bias), alpha = exp(dt * A);
 *       Phase 5: D skip connection, then the silu gate;
 *       decode (Eq. 9): h_t = alpha h_{t-1} + beta prev_Bx + gamma B_t (x) x_t,
 *       y_t = C_t^T h_t.  With lambda = 1 the coefficients are gamma = dt and
 *       beta = (dt - gamma) alpha = 0, which is the update used here.
 *  [P2] same page, section "Kernel details", mamba3_siso_ssd_kernel: the
 *       chunked form (chunk 64, Mamba-2 SSD structure) is mathematically
 *       equivalent to the step-by-step recurrence (oracle_ssd_chunked).
 *  [P2] same page, "How it works", Phase 0 with a general lambda:
 *       gamma = lambda dt, beta = (dt - gamma) alpha, and Eq. 9 with its
 *       beta prev_Bx term (oracle_mamba3_*); "Kernel details",
 *       mamba3_siso_ssd_kernel: the single-SSD form with
 *       scale = gamma + dt_{t+1} (1 - lambda_{t+1}) and a diagonal
 *       correction (oracle_mamba3_chunked).
 *  [P2] same page, "Kernel details", mamba3_mimo_ssd_kernel and
 *       mamba3_mimo_decode_kernel: the rank-R (MIMO) state update,
 *       B x = sum_r B[n,r] x[p,r] and y[p,r] = sum_n state[n,p] C[n,r], and the
 *       rank-flattened chunked form with a block-diagonal correction
 *       (oracle_mamba3_mimo_*).
 *  [P2] same page, "How it works", Phase 1: the angle cumsum
 *       cum_angles = -cumsum(dt * theta), then RoPE applied to B and C
 *       (oracle_mamba3_rope; the complex-valued state of the page's feature
 *       list, "Complex-valued state via data-dependent RoPE").
 *  oracle_scan_bwd: the gradient of the scan above by reverse-mode
 *       differentiation of the same recurrence (the pages mention backward
 *       parity but print no formula; the derivative is pinned by finite
 *       differences of oracle_scan).
 *
 * Readings taken where the pages are silent (each is listed with its reason
 * in the design notes):
 *  - B is discretised by Euler (b = dt * B * x), A by zero-order hold
 *    (a = exp(dt * A)).
 *  - The bias is added before softplus; with softplus off it is still added.
 *  - The gate multiplies after the D skip: y = (sum_n C h + D x) * silu(z),
 *    silu(z) = z / (1 + exp(-z)).
 *  - The prefill state starts at zero unless an initial state is given.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x), written so that no intermediate overflows:
 * for x > 0, log(1 + e^x) = x + log(1 + e^-x). */
static double softplus_d(double x)
{
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double silu_d(double z)
{
    return z / (1.0 + exp(-z));
}

/* The associative combine of two affine maps h -> a h + b applied in
 * sequence, first (a1, b1) then (a2, b2):
 *     (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2).
 * [P1] section "We built the parallel scan": associativity is what lets the
 * sequence be split into pieces. */
void oracle_combine(double a1, double b1, double a2, double b2,
                    double* a_out, double* b_out)
{
    *a_out = a1 * a2;
    *b_out = a2 * b1 + b2;
}

/*
 * Selective scan (Mamba-1 form), one channel at a time.
 *
 *   u, delta, z, y : (batch, dim, seqlen), seqlen contiguous
 *   A              : (dim, dstate)
 *   Bm, Cm         : (batch, ngroups, dstate, seqlen); channel d uses group
 *                    d / (dim / ngroups)
 *   Dskip, delta_bias : (dim,)   (either may be NULL)
 *   z              : may be NULL (no gate)
 *   h0             : (batch, dim, dstate) initial state, or NULL for zero
 *   final_state    : (batch, dim, dstate), may be NULL
 *
 * Per step t, for every state n:
 *   dl = delta + bias;  dl = softplus(dl) if delta_softplus
 *   h_n = exp(dl * A[d,n]) * h_n + dl * B[n,t] * u_t
 *   y_t = sum_n C[n,t] * h_n + D[d] * u_t;   y_t *= silu(z_t) if z given
 */
void oracle_scan(const double* u, const double* delta, const double* A,
                 const double* Bm, const double* Cm, const double* Dskip,
                 const double* z, const double* delta_bias, int delta_softplus,
                 const double* h0, double* y, double* final_state,
                 int batch, int dim, int seqlen, int dstate, int ngroups)
{
    const int dim_per_group = dim / ngroups;
    const long long rows = (long long)batch * dim;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long row = 0; row < rows; ++row) {
        const int b = (int)(row / dim);
        const int d = (int)(row % dim);
        const int g = d / dim_per_group;
        double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int n = 0; n < dstate; ++n)
            h[n] = h0 ? h0[row * dstate + n] : 0.0;
        const size_t io = (size_t)row * (size_t)seqlen;
        const size_t bc = ((size_t)b * ngroups + g) * (size_t)dstate * (size_t)seqlen;
        for (int t = 0; t < seqlen; ++t) {
            double dl = delta[io + t] + (delta_bias ? delta_bias[d] : 0.0);
            if (delta_softplus) dl = softplus_d(dl);
            const double x = u[io + t];
            double acc = 0.0;
            for (int n = 0; n < dstate; ++n) {
                const double a = exp(dl * A[(size_t)d * dstate + n]);
                const double bn = Bm[bc + (size_t)n * seqlen + t];
                const double cn = Cm[bc + (size_t)n * seqlen + t];
                h[n] = a * h[n] + dl * bn * x;
                acc += cn * h[n];
            }
            double out = acc + (Dskip ? Dskip[d] * x : 0.0);
            if (z) out *= silu_d(z[io + t]);
            y[io + t] = out;
        }
        if (final_state)
            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = h[n];
        free(h);
    }
}

/*
 * The same scan evaluated piecewise, to pin the split-and-combine algorithm
 * against the sequential definition.  The sequence is cut at the
 * npieces - 1 increasing positions in `cuts` (0 < cut < seqlen).  Each piece
 * is first scanned from a zero state, giving its aggregate map
 * (prod a, h_end); the carried-in state of piece k is the exclusive
 * o-combination of the aggregates of pieces 0..k-1 applied to h0; each piece
 * is then scanned again from its carried-in state to produce y.
 * Arguments otherwise as oracle_scan.
 */
void oracle_scan_pieces(const double* u, const double* delta, const double* A,
                        const double* Bm, const double* Cm, const double* Dskip,
                        const double* z, const double* delta_bias, int delta_softplus,
                        const double* h0, double* y, double* final_state,
                        int batch, int dim, int seqlen, int dstate, int ngroups,
                        const int* cuts, int ncuts)
{
    const int dim_per_group = dim / ngroups;
    const long long rows = (long long)batch * dim;
    const int npieces = ncuts + 1;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long row = 0; row < rows; ++row) {
        const int b = (int)(row / dim);
        const int d = (int)(row % dim);
        const int g = d / dim_per_group;
        const size_t io = (size_t)row * (size_t)seqlen;
        const size_t bc = ((size_t)b * ngroups + g) * (size_t)dstate * (size_t)seqlen;
        double* agg_a = (double*)malloc(sizeof(double) * (size_t)npieces * dstate);
        double* agg_b = (double*)malloc(sizeof(double) * (size_t)npieces * dstate);
        double* carry = (double*)malloc(sizeof(double) * (size_t)dstate);
        /* pass 1: aggregate of every piece, from a zero state */
        for (int k = 0; k < npieces; ++k) {
            const int t0 = k == 0 ? 0 : cuts[k - 1];
            const int t1 = k == npieces - 1 ? seqlen : cuts[k];
            for (int n = 0; n < dstate; ++n) {
                double pa = 1.0, hb = 0.0;
                for (int t = t0; t < t1; ++t) {
                    double dl = delta[io + t] + (delta_bias ? delta_bias[d] : 0.0);
                    if (delta_softplus) dl = softplus_d(dl);
                    const double a = exp(dl * A[(size_t)d * dstate + n]);
                    const double bt = dl * Bm[bc + (size_t)n * seqlen + t] * u[io + t];
                    oracle_combine(pa, hb, a, bt, &pa, &hb);
                }
                agg_a[k * dstate + n] = pa;
                agg_b[k * dstate + n] = hb;
            }
        }
        /* pass 2: carried-in state of every piece, then the piece's outputs */
        for (int n = 0; n < dstate; ++n) carry[n] = h0 ? h0[row * dstate + n] : 0.0;
        for (int k = 0; k < npieces; ++k) {
            const int t0 = k == 0 ? 0 : cuts[k - 1];
            const int t1 = k == npieces - 1 ? seqlen : cuts[k];
            double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
            memcpy(h, carry, sizeof(double) * (size_t)dstate);
            for (int t = t0; t < t1; ++t) {
                double dl = delta[io + t] + (delta_bias ? delta_bias[d] : 0.0);
                if (delta_softplus) dl = softplus_d(dl);
                const double x = u[io + t];
                double acc = 0.0;
                for (int n = 0; n < dstate; ++n) {
                    const double a = exp(dl * A[(size_t)d * dstate + n]);
                    h[n] = a * h[n] + dl * Bm[bc + (size_t)n * seqlen + t] * x;
                    acc += Cm[bc + (size_t)n * seqlen + t] * h[n];
                }
                double out = acc + (Dskip ? Dskip[d] * x : 0.0);
                if (z) out *= silu_d(z[io + t]);
                y[io + t] = out;
            }
            free(h);
            /* carry into the next piece: (1, carry) o aggregate(k) */
            for (int n = 0; n < dstate; ++n) {
                double na, nb;
                oracle_combine(1.0, carry[n], agg_a[k * dstate + n], agg_b[k * dstate + n],
                               &na, &nb);
                carry[n] = nb;
            }
        }
        if (final_state)
            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = carry[n];
        free(agg_a);
        free(agg_b);
        free(carry);
    }
}

/*
 * Scalar-A-per-head SSD, evaluated as the plain recurrence.
 *
 *   x, y        : (batch, seqlen, nheads, headdim)
 *   dt          : (batch, seqlen, nheads)   (already discretised: > 0)
 *   A_head      : (nheads,)
 *   Bm, Cm      : (batch, seqlen, ngroups, dstate); head h uses group
 *                 h / (nheads / ngroups)
 *   h0          : (batch, nheads, headdim, dstate) or NULL for zero
 *   final_state : (batch, nheads, headdim, dstate), may be NULL
 *
 * Per step t:  S[p,n] = exp(dt_t A_h) S[p,n] + dt_t B_t[n] x_t[p],
 *              y_t[p] = sum_n C_t[n] S[p,n].
 */
void oracle_ssd_recurrence(const double* x, const double* dt, const double* A_head,
                           const double* Bm, const double* Cm, const double* h0,
                           double* y, double* final_state,
                           int batch, int seqlen, int nheads, int headdim, int dstate,
                           int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(dynamic, 8)
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        double* S = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int n = 0; n < dstate; ++n) S[n] = h0 ? h0[row * dstate + n] : 0.0;
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double dtv = dt[bt * nheads + h];
            const double a = exp(dtv * A_head[h]);
            const double xv = x[(bt * nheads + h) * headdim + p];
            const double* Bt = Bm + (bt * ngroups + g) * dstate;
            const double* Ct = Cm + (bt * ngroups + g) * dstate;
            double acc = 0.0;
            for (int n = 0; n < dstate; ++n) {
                S[n] = a * S[n] + dtv * Bt[n] * xv;
                acc += Ct[n] * S[n];
            }
            y[(bt * nheads + h) * headdim + p] = acc;
        }
        if (final_state)
            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = S[n];
        free(S);
    }
}

/*
 * The same SSD evaluated by the chunked algorithm, in fp64, as plain loops.
 * [P2] "Kernel details", mamba3_siso_ssd_kernel: the chunked (Mamba-2 SSD)
 * structure, stated there to be mathematically equivalent to the recurrence.
 * For each chunk c of `chunk` steps (the last one may be shorter):
 *   cs_i      = sum_{j <= i} dt_j A_h                 (within the chunk)
 *   G[i,j]    = sum_n C_i[n] B_j[n]
 *   M[i,j]    = G[i,j] exp(cs_i - cs_j)   for j <= i, else 0
 *   Y_diag    = M (dt o x)
 *   Y_off[i]  = exp(cs_i) sum_n C_i[n] S_prev[:, n]
 *   S_chunk   = sum_j exp(cs_last - cs_j) dt_j x_j (x) B_j
 *   S_prev    = exp(cs_last) S_prev + S_chunk
 * Arguments as oracle_ssd_recurrence.
 */
void oracle_ssd_chunked(const double* x, const double* dt, const double* A_head,
                        const double* Bm, const double* Cm, const double* h0,
                        double* y, double* final_state,
                        int batch, int seqlen, int nheads, int headdim, int dstate,
                        int ngroups, int chunk)
{
    const int heads_per_group = nheads / ngroups;
    const long long units = (long long)batch * nheads;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long unit = 0; unit < units; ++unit) {
        const int h = (int)(unit % nheads);
        const int b = (int)(unit / nheads);
        const int g = h / heads_per_group;
        const double Ah = A_head[h];
        double* S = (double*)calloc((size_t)headdim * dstate, sizeof(double));
        double* cs = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* M = (double*)malloc(sizeof(double) * (size_t)chunk * chunk);
        double* Sc = (double*)malloc(sizeof(double) * (size_t)headdim * dstate);
        if (h0)
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n)
                    S[(size_t)p * dstate + n] =
                        h0[(((size_t)b * nheads + h) * headdim + p) * dstate + n];
        for (int t0 = 0; t0 < seqlen; t0 += chunk) {
            const int q = seqlen - t0 < chunk ? seqlen - t0 : chunk;
#define DT(i) dt[((size_t)b * seqlen + t0 + (i)) * nheads + h]
#define XV(i, p) x[(((size_t)b * seqlen + t0 + (i)) * nheads + h) * headdim + (p)]
#define BV(i, n) Bm[(((size_t)b * seqlen + t0 + (i)) * ngroups + g) * dstate + (n)]
#define CV(i, n) Cm[(((size_t)b * seqlen + t0 + (i)) * ngroups + g) * dstate + (n)]
            /* cumulative log-decay inside the chunk */
            double run = 0.0;
            for (int i = 0; i < q; ++i) {
                run += DT(i) * Ah;
                cs[i] = run;
            }
            /* M = (C B^T) masked by the causal decay exp(cs_i - cs_j) */
            for (int i = 0; i < q; ++i)
                for (int j = 0; j < q; ++j) {
                    double m = 0.0;
                    if (j <= i) {
                        double gij = 0.0;
                        for (int n = 0; n < dstate; ++n) gij += CV(i, n) * BV(j, n);
                        m = gij * exp(cs[i] - cs[j]);
                    }
                    M[(size_t)i * chunk + j] = m;
                }
            /* outputs: diagonal block plus the contribution of the carried state */
            for (int i = 0; i < q; ++i)
                for (int p = 0; p < headdim; ++p) {
                    double yd = 0.0;
                    for (int j = 0; j <= i; ++j) yd += M[(size_t)i * chunk + j] * DT(j) * XV(j, p);
                    double yo = 0.0;
                    for (int n = 0; n < dstate; ++n) yo += CV(i, n) * S[(size_t)p * dstate + n];
                    yo *= exp(cs[i]);
                    y[(((size_t)b * seqlen + t0 + i) * nheads + h) * headdim + p] = yd + yo;
                }
            /* state produced inside the chunk, then the inter-chunk recurrence */
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n) {
                    double s = 0.0;
                    for (int j = 0; j < q; ++j)
                        s += exp(cs[q - 1] - cs[j]) * DT(j) * XV(j, p) * BV(j, n);
                    Sc[(size_t)p * dstate + n] = s;
                }
            const double decay = exp(cs[q - 1]);
            for (size_t k = 0; k < (size_t)headdim * dstate; ++k) S[k] = decay * S[k] + Sc[k];
#undef DT
#undef XV
#undef BV
#undef CV
        }
        if (final_state)
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n)
                    final_state[(((size_t)b * nheads + h) * headdim + p) * dstate + n] =
                        S[(size_t)p * dstate + n];
        free(S);
        free(cs);
        free(M);
        free(Sc);
    }
}

/*
 * One decode step, updating `state` in place.
 * [P2] "How it works", decode via step(), Eq. 9 with lambda = 1.
 *
 *   state : (batch, nheads, headdim, dstate), read and overwritten
 *   x, z, y : (batch, nheads, headdim); z may be NULL
 *   dt    : (batch, nheads);  A, D : (nheads,); D may be NULL
 *   Bm, Cm : (batch, ngroups, dstate)
 *
 *   alpha = exp(dt A_h);  s[n] = alpha s[n] + dt x B[n];
 *   y = sum_n C[n] s[n] + D_h x;  y *= silu(z) if z given.
 */
void oracle_decode_step(double* state, const double* x, const double* dt,
                        const double* A, const double* Bm, const double* Cm,
                        const double* Dskip, const double* z, double* y,
                        int batch, int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(static)
    for (long long row = 0; row < rows; ++row) {
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        const double dtv = dt[(size_t)b * nheads + h];
        const double alpha = exp(dtv * A[h]);
        const double xv = x[row];
        const double* Bt = Bm + ((size_t)b * ngroups + g) * dstate;
        const double* Ct = Cm + ((size_t)b * ngroups + g) * dstate;
        double* s = state + (size_t)row * dstate;
        double acc = 0.0;
        for (int n = 0; n < dstate; ++n) {
            s[n] = alpha * s[n] + dtv * xv * Bt[n];
            acc += Ct[n] * s[n];
        }
        double out = acc + (Dskip ? Dskip[h] * xv : 0.0);
        if (z) out *= silu_d(z[row]);
        y[row] = out;
    }
}

/* Number of OpenMP threads the oracle's parallel loops use. */
/*
 * Mamba-3 SISO recurrence, one step after another.
 * [P2] "How it works", Phase 0 (alpha = exp(dt A), gamma = lambda dt,
 * beta = (dt - gamma) alpha) and decode via step(), Eq. 9:
 *   h_t = alpha_t h_{t-1} + beta_t (B_{t-1} (x) x_{t-1}) + gamma_t (B_t (x) x_t),
 *   y_t = C_t^T h_t.
 * dt and lambda are taken as given (dt after softplus, lambda after sigmoid).
 * The term before the first step uses h0 (NULL: 0) and the previous token's
 * B and x, prev_B (batch, ngroups, dstate) and prev_x (batch, nheads,
 * headdim) (NULL: no previous token).
 *
 *   x, y : (batch, seqlen, nheads, headdim);  dt, lam : (batch, seqlen, nheads)
 *   A_head : (nheads,);  Bm, Cm : (batch, seqlen, ngroups, dstate)
 *   h0, final_state : (batch, nheads, headdim, dstate); either may be NULL
 */
void oracle_mamba3_recurrence(const double* x, const double* dt, const double* lam,
                              const double* A_head, const double* Bm, const double* Cm,
                              const double* h0, const double* prev_B, const double* prev_x,
                              double* y, double* final_state, int batch, int seqlen, int nheads,
                              int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(dynamic, 8)
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        double* S = (double*)malloc(sizeof(double) * (size_t)dstate);
        double* Bprev = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int n = 0; n < dstate; ++n) {
            S[n] = h0 ? h0[row * dstate + n] : 0.0;
            Bprev[n] = prev_B ? prev_B[((size_t)b * ngroups + g) * dstate + n] : 0.0;
        }
        double xprev = prev_x ? prev_x[row] : 0.0;
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double dtv = dt[bt * nheads + h];
            const double alpha = exp(dtv * A_head[h]);
            const double gamma = lam[bt * nheads + h] * dtv;
            const double beta = (dtv - gamma) * alpha;
            const double xv = x[(bt * nheads + h) * headdim + p];
            const double* Bt = Bm + (bt * ngroups + g) * dstate;
            const double* Ct = Cm + (bt * ngroups + g) * dstate;
            double acc = 0.0;
            for (int n = 0; n < dstate; ++n) {
                S[n] = alpha * S[n] + beta * Bprev[n] * xprev + gamma * Bt[n] * xv;
                acc += Ct[n] * S[n];
            }
            y[(bt * nheads + h) * headdim + p] = acc;
            for (int n = 0; n < dstate; ++n) Bprev[n] = Bt[n];
            xprev = xv;
        }
        if (final_state)
            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = S[n];
        free(S);
        free(Bprev);
    }
}

/*
 * Mamba-3 SISO, chunked single-SSD form.
 * [P2] "Kernel details", mamba3_siso_ssd_kernel: the Mamba-2 chunked SSD
 * (as oracle_ssd_chunked) with x weighted by
 *   scale_s = gamma_s + dt_{s+1} (1 - lambda_{s+1})   (0 past the last step)
 * instead of dt_s, and a diagonal correction: on the diagonal (s = t) the
 * weight is gamma_t alone, since the beta_{t+1} part of step s reaches the
 * state only at step t + 1.  The carried state is therefore the true state
 * plus the not-yet-applied dt_{t+1} (1 - lambda_{t+1}) (B_t (x) x_t) of the
 * chunk's last step, which is exactly what the next chunk's decay turns into
 * its beta term.  Before the first step that pending term comes from the
 * previous token: S = h0 + dt_0 (1 - lambda_0) (prev_B (x) prev_x).
 * Arguments as oracle_mamba3_recurrence, plus the chunk length.
 */
void oracle_mamba3_chunked(const double* x, const double* dt, const double* lam,
                           const double* A_head, const double* Bm, const double* Cm,
                           const double* h0, const double* prev_B, const double* prev_x,
                           double* y, double* final_state, int batch, int seqlen, int nheads,
                           int headdim, int dstate, int ngroups, int chunk)
{
    const int heads_per_group = nheads / ngroups;
    const long long units = (long long)batch * nheads;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long unit = 0; unit < units; ++unit) {
        const int h = (int)(unit % nheads);
        const int b = (int)(unit / nheads);
        const int g = h / heads_per_group;
        const double Ah = A_head[h];
        double* S = (double*)calloc((size_t)headdim * dstate, sizeof(double));
        double* cs = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* w = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* wd = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* M = (double*)malloc(sizeof(double) * (size_t)chunk * chunk);
        double* Sc = (double*)malloc(sizeof(double) * (size_t)headdim * dstate);
#define DTA(t) dt[((size_t)b * seqlen + (t)) * nheads + h]
#define LMA(t) lam[((size_t)b * seqlen + (t)) * nheads + h]
        for (int p = 0; p < headdim; ++p)
            for (int n = 0; n < dstate; ++n) {
                double s0 = h0 ? h0[(((size_t)b * nheads + h) * headdim + p) * dstate + n] : 0.0;
                if (prev_B && prev_x && seqlen > 0)
                    s0 += DTA(0) * (1.0 - LMA(0)) *
                          prev_B[((size_t)b * ngroups + g) * dstate + n] *
                          prev_x[((size_t)b * nheads + h) * headdim + p];
                S[(size_t)p * dstate + n] = s0;
            }
        for (int t0 = 0; t0 < seqlen; t0 += chunk) {
            const int q = seqlen - t0 < chunk ? seqlen - t0 : chunk;
#define XV(i, p) x[(((size_t)b * seqlen + t0 + (i)) * nheads + h) * headdim + (p)]
#define BV(i, n) Bm[(((size_t)b * seqlen + t0 + (i)) * ngroups + g) * dstate + (n)]
#define CV(i, n) Cm[(((size_t)b * seqlen + t0 + (i)) * ngroups + g) * dstate + (n)]
            double run = 0.0;
            for (int i = 0; i < q; ++i) {
                const int t = t0 + i;
                run += DTA(t) * Ah;
                cs[i] = run;
                wd[i] = LMA(t) * DTA(t);  /* gamma_t: the diagonal weight */
                w[i] = wd[i] + (t + 1 < seqlen ? DTA(t + 1) * (1.0 - LMA(t + 1)) : 0.0);
            }
            for (int i = 0; i < q; ++i)
                for (int j = 0; j < q; ++j) {
                    double m = 0.0;
                    if (i >= j) {
                        double gij = 0.0;
                        for (int n = 0; n < dstate; ++n) gij += CV(i, n) * BV(j, n);
                        m = gij * exp(cs[i] - cs[j]) * (j < i ? w[j] : wd[j]);
                    }
                    M[(size_t)i * chunk + j] = m;
                }
            for (int i = 0; i < q; ++i)
                for (int p = 0; p < headdim; ++p) {
                    double yd = 0.0;
                    for (int j = 0; j <= i; ++j) yd += M[(size_t)i * chunk + j] * XV(j, p);
                    double yo = 0.0;
                    for (int n = 0; n < dstate; ++n) yo += CV(i, n) * S[(size_t)p * dstate + n];
                    yo = exp(cs[i]) * yo;
                    y[(((size_t)b * seqlen + t0 + i) * nheads + h) * headdim + p] = yd + yo;
                }
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n) {
                    double s = 0.0;
                    for (int j = 0; j < q; ++j)
                        s += exp(cs[q - 1] - cs[j]) * w[j] * XV(j, p) * BV(j, n);
                    Sc[(size_t)p * dstate + n] = s;
                }
            const double decay = exp(cs[q - 1]);
            for (size_t k = 0; k < (size_t)headdim * dstate; ++k) S[k] = decay * S[k] + Sc[k];
#undef XV
#undef BV
#undef CV
        }
#undef DTA
#undef LMA
        if (final_state)
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n)
                    final_state[(((size_t)b * nheads + h) * headdim + p) * dstate + n] =
                        S[(size_t)p * dstate + n];
        free(S);
        free(cs);
        free(w);
        free(wd);
        free(M);
        free(Sc);
    }
}

/*
 * One Mamba-3 SISO decode step, updating `state` in place.
 * [P2] "How it works", decode via step(), Eq. 9, and Phase 5 (D skip, silu).
 *
 *   alpha = exp(dt A_h), gamma = lambda dt, beta = (dt - gamma) alpha;
 *   s = alpha s + beta prev_B (x) prev_x + gamma B (x) x;
 *   y = sum_n C s + D_h x;  y *= silu(z) if z given.
 * prev_B (batch, ngroups, dstate) and prev_x (batch, nheads, headdim) are the
 * previous token's B and x; dt, lam (batch, nheads); other arguments as
 * oracle_decode_step.
 */
void oracle_mamba3_decode_step(double* state, const double* prev_B, const double* prev_x,
                               const double* x, const double* dt, const double* lam,
                               const double* A, const double* Bm, const double* Cm,
                               const double* Dskip, const double* z, double* y, int batch,
                               int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(static)
    for (long long row = 0; row < rows; ++row) {
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        const double dtv = dt[(size_t)b * nheads + h];
        const double alpha = exp(A[h] * dtv);
        const double gamma = lam[(size_t)b * nheads + h] * dtv;
        const double beta = alpha * (dtv - gamma);
        const double xv = x[row], xp = prev_x[row];
        const double* Bt = Bm + ((size_t)b * ngroups + g) * dstate;
        const double* Bp = prev_B + ((size_t)b * ngroups + g) * dstate;
        const double* Ct = Cm + ((size_t)b * ngroups + g) * dstate;
        double* s = state + row * dstate;
        double acc = 0.0;
        for (int n = 0; n < dstate; ++n) {
            s[n] = alpha * s[n] + beta * Bp[n] * xp + gamma * Bt[n] * xv;
            acc += Ct[n] * s[n];
        }
        double out = acc + (Dskip ? xv * Dskip[h] : 0.0);
        if (z) out *= silu_d(z[row]);
        y[row] = out;
    }
}

/*
 * Mamba-3 MIMO (rank R) recurrence.
 * [P2] "How it works" (Phase 0, Eq. 9) with the rank-R terms of "Kernel
 * details", mamba3_mimo_decode_kernel:
 *   BX_t[n,p] = sum_r B_t[n,r] x_t[p,r]
 *   h_t = alpha_t h_{t-1} + beta_t BX_{t-1} + gamma_t BX_t
 *   y_t[p,r] = sum_n h_t[n,p] C_t[n,r]
 * Layouts (rank inside the time position):
 *   x, y : (batch, seqlen, R, nheads, headdim);  dt, lam : (batch, seqlen, nheads)
 *   Bm, Cm : (batch, seqlen, R, ngroups, dstate);  A_head : (nheads,)
 *   h0, final_state : (batch, nheads, headdim, dstate); either may be NULL
 *   prev_B : (batch, R, ngroups, dstate), prev_x : (batch, R, nheads, headdim):
 *   the token before the first (NULL: none).
 */
void oracle_mamba3_mimo_recurrence(const double* x, const double* dt, const double* lam,
                                   const double* A_head, const double* Bm, const double* Cm,
                                   const double* h0, const double* prev_B, const double* prev_x,
                                   double* y, double* final_state, int batch, int seqlen,
                                   int rank, int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(dynamic, 8)
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        double* S = (double*)malloc(sizeof(double) * (size_t)dstate);
        double* BXp = (double*)malloc(sizeof(double) * (size_t)dstate);
        double* BX = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int n = 0; n < dstate; ++n) {
            S[n] = h0 ? h0[row * dstate + n] : 0.0;
            double bx = 0.0;
            if (prev_B && prev_x)
                for (int r = 0; r < rank; ++r)
                    bx += prev_B[(((size_t)b * rank + r) * ngroups + g) * dstate + n] *
                          prev_x[(((size_t)b * rank + r) * nheads + h) * headdim + p];
            BXp[n] = bx;
        }
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double dtv = dt[bt * nheads + h];
            const double alpha = exp(dtv * A_head[h]);
            const double gamma = lam[bt * nheads + h] * dtv;
            const double beta_t = (dtv - gamma) * alpha;
            for (int n = 0; n < dstate; ++n) {
                double bx = 0.0;
                for (int r = 0; r < rank; ++r)
                    bx += Bm[((bt * rank + r) * ngroups + g) * dstate + n] *
                          x[((bt * rank + r) * nheads + h) * headdim + p];
                BX[n] = bx;
                S[n] = alpha * S[n] + beta_t * BXp[n] + gamma * bx;
            }
            for (int r = 0; r < rank; ++r) {
                double acc = 0.0;
                for (int n = 0; n < dstate; ++n)
                    acc += Cm[((bt * rank + r) * ngroups + g) * dstate + n] * S[n];
                y[((bt * rank + r) * nheads + h) * headdim + p] = acc;
            }
            for (int n = 0; n < dstate; ++n) BXp[n] = BX[n];
        }
        if (final_state)
            for (int n = 0; n < dstate; ++n) final_state[row * dstate + n] = S[n];
        free(S);
        free(BXp);
        free(BX);
    }
}

/*
 * Mamba-3 MIMO, rank-flattened chunked form.
 * [P2] "Kernel details", mamba3_mimo_ssd_kernel: the (step, rank) pairs of a
 * chunk are taken as chunk * R sub-tokens, and the chunked single-SSD form of
 * oracle_mamba3_chunked runs over them: sub-tokens share the decay and the
 * weights of their step (scale off the diagonal, gamma on it), and the
 * causal mask is block-lower-triangular -- a sub-token sees every sub-token of
 * its own step (the block-diagonal part, weight gamma) and of earlier steps.
 * `chunk` counts steps.  Arguments as oracle_mamba3_mimo_recurrence.
 */
void oracle_mamba3_mimo_chunked(const double* x, const double* dt, const double* lam,
                                const double* A_head, const double* Bm, const double* Cm,
                                const double* h0, const double* prev_B, const double* prev_x,
                                double* y, double* final_state, int batch, int seqlen, int rank,
                                int nheads, int headdim, int dstate, int ngroups, int chunk)
{
    const int heads_per_group = nheads / ngroups;
    const long long units = (long long)batch * nheads;
    const int qmax = chunk * rank;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long unit = 0; unit < units; ++unit) {
        const int h = (int)(unit % nheads);
        const int b = (int)(unit / nheads);
        const int g = h / heads_per_group;
        const double Ah = A_head[h];
        double* S = (double*)calloc((size_t)headdim * dstate, sizeof(double));
        double* cs = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* w = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* wd = (double*)malloc(sizeof(double) * (size_t)chunk);
        double* M = (double*)malloc(sizeof(double) * (size_t)qmax * qmax);
        double* Sc = (double*)malloc(sizeof(double) * (size_t)headdim * dstate);
#define DTM(t) dt[((size_t)b * seqlen + (t)) * nheads + h]
#define LMM(t) lam[((size_t)b * seqlen + (t)) * nheads + h]
        for (int p = 0; p < headdim; ++p)
            for (int n = 0; n < dstate; ++n) {
                double s0 = h0 ? h0[(((size_t)b * nheads + h) * headdim + p) * dstate + n] : 0.0;
                if (prev_B && prev_x && seqlen > 0)
                    for (int r = 0; r < rank; ++r)
                        s0 += DTM(0) * (1.0 - LMM(0)) *
                              prev_B[(((size_t)b * rank + r) * ngroups + g) * dstate + n] *
                              prev_x[(((size_t)b * rank + r) * nheads + h) * headdim + p];
                S[(size_t)p * dstate + n] = s0;
            }
        for (int t0 = 0; t0 < seqlen; t0 += chunk) {
            const int q = seqlen - t0 < chunk ? seqlen - t0 : chunk;
            const int qs = q * rank;  /* sub-tokens i = (step i / R, rank i % R) */
#define XS(i, p) x[((((size_t)b * seqlen + t0) * rank + (i)) * nheads + h) * headdim + (p)]
#define BS(i, n) Bm[((((size_t)b * seqlen + t0) * rank + (i)) * ngroups + g) * dstate + (n)]
#define CS(i, n) Cm[((((size_t)b * seqlen + t0) * rank + (i)) * ngroups + g) * dstate + (n)]
            double run = 0.0;
            for (int k = 0; k < q; ++k) {
                const int t = t0 + k;
                run += DTM(t) * Ah;
                cs[k] = run;
                wd[k] = LMM(t) * DTM(t);
                w[k] = wd[k] + (t + 1 < seqlen ? DTM(t + 1) * (1.0 - LMM(t + 1)) : 0.0);
            }
            for (int i = 0; i < qs; ++i)
                for (int j = 0; j < qs; ++j) {
                    const int si = i / rank, sj = j / rank;
                    double m = 0.0;
                    if (sj <= si) {
                        double gij = 0.0;
                        for (int n = 0; n < dstate; ++n) gij += CS(i, n) * BS(j, n);
                        m = gij * exp(cs[si] - cs[sj]) * (sj < si ? w[sj] : wd[sj]);
                    }
                    M[(size_t)i * qmax + j] = m;
                }
            for (int i = 0; i < qs; ++i)
                for (int p = 0; p < headdim; ++p) {
                    double yd = 0.0;
                    for (int j = 0; j < qs; ++j) yd += M[(size_t)i * qmax + j] * XS(j, p);
                    double yo = 0.0;
                    for (int n = 0; n < dstate; ++n) yo += CS(i, n) * S[(size_t)p * dstate + n];
                    y[((((size_t)b * seqlen + t0) * rank + i) * nheads + h) * headdim + p] =
                        yd + exp(cs[i / rank]) * yo;
                }
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n) {
                    double s = 0.0;
                    for (int j = 0; j < qs; ++j)
                        s += exp(cs[q - 1] - cs[j / rank]) * w[j / rank] * XS(j, p) * BS(j, n);
                    Sc[(size_t)p * dstate + n] = s;
                }
            const double decay = exp(cs[q - 1]);
            for (size_t k = 0; k < (size_t)headdim * dstate; ++k) S[k] = decay * S[k] + Sc[k];
#undef XS
#undef BS
#undef CS
        }
#undef DTM
#undef LMM
        if (final_state)
            for (int p = 0; p < headdim; ++p)
                for (int n = 0; n < dstate; ++n)
                    final_state[(((size_t)b * nheads + h) * headdim + p) * dstate + n] =
                        S[(size_t)p * dstate + n];
        free(S);
        free(cs);
        free(w);
        free(wd);
        free(M);
        free(Sc);
    }
}

/*
 * One Mamba-3 MIMO decode step, updating `state` in place.
 * [P2] "Kernel details", mamba3_mimo_decode_kernel, with Phase 5 per rank:
 *   s = alpha s + beta sum_r prev_B[.,r] (x) prev_x[.,r] + gamma sum_r B[.,r] (x) x[.,r]
 *   y[p,r] = (sum_n C[n,r] s[p,n] + D_h x[p,r]) * silu(z[p,r])
 * x, z, y, prev_x : (batch, R, nheads, headdim); B, C, prev_B :
 * (batch, R, ngroups, dstate); dt, lam : (batch, nheads); A, D : (nheads,).
 */
void oracle_mamba3_mimo_decode_step(double* state, const double* prev_B, const double* prev_x,
                                    const double* x, const double* dt, const double* lam,
                                    const double* A, const double* Bm, const double* Cm,
                                    const double* Dskip, const double* z, double* y, int batch,
                                    int rank, int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const long long rows = (long long)batch * nheads * headdim;
#pragma omp parallel for schedule(static)
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        const double dtv = dt[(size_t)b * nheads + h];
        const double alpha = exp(A[h] * dtv);
        const double gamma = lam[(size_t)b * nheads + h] * dtv;
        const double beta = alpha * (dtv - gamma);
        double* s = state + row * dstate;
        for (int n = 0; n < dstate; ++n) {
            double bx = 0.0, bxp = 0.0;
            for (int r = 0; r < rank; ++r) {
                const size_t ib = (((size_t)b * rank + r) * ngroups + g) * dstate + n;
                const size_t ix = (((size_t)b * rank + r) * nheads + h) * headdim + p;
                bx += Bm[ib] * x[ix];
                bxp += prev_B[ib] * prev_x[ix];
            }
            s[n] = alpha * s[n] + beta * bxp + gamma * bx;
        }
        for (int r = 0; r < rank; ++r) {
            const size_t ix = (((size_t)b * rank + r) * nheads + h) * headdim + p;
            const double* Cr = Cm + (((size_t)b * rank + r) * ngroups + g) * dstate;
            double acc = 0.0;
            for (int n = 0; n < dstate; ++n) acc += Cr[n] * s[n];
            double out = acc + (Dskip ? Dskip[h] * x[ix] : 0.0);
            if (z) out *= silu_d(z[ix]);
            y[ix] = out;
        }
    }
}

/*
 * Gradient of oracle_scan for the loss  sum_t dy . y + sum dfinal . final_state
 * (dfinal may be NULL), by differentiating the recurrence in reverse:
 *   lambda_t = dL/dh_t = dy0_t C_t + a_{t+1} lambda_{t+1},   dy0_t = dy_t silu(z_t)
 *   dC_t += dy0_t h_t;  dB_t += lambda_t dl_t u_t;  du_t = dy0_t D + sum_n lambda_t dl_t B_t
 *   d dl_t = sum_n lambda_t (h_{t-1} A a_t + B_t u_t);  dA += lambda_t h_{t-1} a_t dl_t
 *   ddelta_t = d dl_t * sigmoid(delta_t + bias) (softplus) or d dl_t;  dbias += ddelta_t
 *   dz_t = dy_t y0_t silu'(z_t);  dD += dy0_t u_t;  dh0 = a_0 lambda_0.
 * Serial over rows (dB, dC, dA, dD, dbias are sums over several rows), for
 * small problems.  Arguments as oracle_scan plus dy (batch, dim, seqlen) and
 * dfinal (batch, dim, dstate) in, and out: du, ddelta, dz (batch, dim,
 * seqlen), dA (dim, dstate), dB, dC (batch, ngroups, dstate, seqlen), dD,
 * dbias (dim), dh0 (batch, dim, dstate).  dz, dD, dbias, dh0 may be NULL
 * (their inputs absent or the gradient not wanted).
 */
void oracle_scan_bwd(const double* u, const double* delta, const double* A,
                     const double* Bm, const double* Cm, const double* Dskip,
                     const double* z, const double* delta_bias, int delta_softplus,
                     const double* h0, const double* dy, const double* dfinal,
                     double* du, double* ddelta, double* dA, double* dB, double* dC,
                     double* dD, double* dz, double* dbias, double* dh0,
                     int batch, int dim, int seqlen, int dstate, int ngroups)
{
    const int dim_per_group = dim / ngroups;
    memset(dA, 0, sizeof(double) * (size_t)dim * dstate);
    memset(dB, 0, sizeof(double) * (size_t)batch * ngroups * dstate * seqlen);
    memset(dC, 0, sizeof(double) * (size_t)batch * ngroups * dstate * seqlen);
    if (dD) memset(dD, 0, sizeof(double) * (size_t)dim);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)dim);
    double* H = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * dstate);  /* h_{t-1} at t */
    double* Aa = (double*)malloc(sizeof(double) * (size_t)seqlen * dstate);        /* a_t */
    double* dl = (double*)malloc(sizeof(double) * (size_t)seqlen);
    double* pre = (double*)malloc(sizeof(double) * (size_t)seqlen);  /* delta + bias */
    double* y0 = (double*)malloc(sizeof(double) * (size_t)seqlen);
    double* lam = (double*)malloc(sizeof(double) * (size_t)dstate);
    for (long long row = 0; row < (long long)batch * dim; ++row) {
        const int b = (int)(row / dim);
        const int d = (int)(row % dim);
        const int g = d / dim_per_group;
        const size_t io = (size_t)row * (size_t)seqlen;
        const size_t bc = ((size_t)b * ngroups + g) * (size_t)dstate * (size_t)seqlen;
        const double Dd = Dskip ? Dskip[d] : 0.0;
        /* forward, keeping every state */
        for (int n = 0; n < dstate; ++n) H[n] = h0 ? h0[row * dstate + n] : 0.0;
        for (int t = 0; t < seqlen; ++t) {
            pre[t] = delta[io + t] + (delta_bias ? delta_bias[d] : 0.0);
            dl[t] = delta_softplus ? softplus_d(pre[t]) : pre[t];
            double acc = 0.0;
            for (int n = 0; n < dstate; ++n) {
                const double a = exp(dl[t] * A[(size_t)d * dstate + n]);
                Aa[(size_t)t * dstate + n] = a;
                const double hn = a * H[(size_t)t * dstate + n] +
                                  dl[t] * Bm[bc + (size_t)n * seqlen + t] * u[io + t];
                H[(size_t)(t + 1) * dstate + n] = hn;
                acc += Cm[bc + (size_t)n * seqlen + t] * hn;
            }
            y0[t] = acc + Dd * u[io + t];
        }
        /* reverse */
        for (int n = 0; n < dstate; ++n) lam[n] = dfinal ? dfinal[row * dstate + n] : 0.0;
        for (int t = seqlen - 1; t >= 0; --t) {
            const double ut = u[io + t];
            double dy0 = dy[io + t];
            if (z) {
                const double zt = z[io + t];
                const double sg = 1.0 / (1.0 + exp(-zt));
                if (dz) dz[io + t] = dy0 * y0[t] * sg * (1.0 + zt * (1.0 - sg));
                dy0 *= zt * sg;
            }
            double dut = dy0 * Dd;
            if (dD) dD[d] += dy0 * ut;
            double ddl = 0.0;
            for (int n = 0; n < dstate; ++n) {
                const size_t ib = bc + (size_t)n * seqlen + t;
                const double a = Aa[(size_t)t * dstate + n];
                const double hprev = H[(size_t)t * dstate + n];
                lam[n] += dy0 * Cm[ib];
                dC[ib] += dy0 * H[(size_t)(t + 1) * dstate + n];
                dB[ib] += lam[n] * dl[t] * ut;
                dA[(size_t)d * dstate + n] += lam[n] * hprev * a * dl[t];
                ddl += lam[n] * (hprev * a * A[(size_t)d * dstate + n] + Bm[ib] * ut);
                dut += lam[n] * dl[t] * Bm[ib];
                lam[n] *= a;
            }
            du[io + t] = dut;
            const double dd = delta_softplus ? ddl / (1.0 + exp(-pre[t])) : ddl;
            ddelta[io + t] = dd;
            if (dbias) dbias[d] += dd;
        }
        if (dh0)
            for (int n = 0; n < dstate; ++n) dh0[row * dstate + n] = lam[n];
    }
    free(H);
    free(Aa);
    free(dl);
    free(pre);
    free(y0);
    free(lam);
}

/*
 * Gradient of oracle_ssd_recurrence for the loss  sum dy . y + sum dfinal .
 * final_state (dfinal may be NULL), by differentiating the recurrence in
 * reverse, with Lambda_t = dL/dS_t (a headdim x dstate matrix per head):
 *   Lambda_t = dy_t (outer) C_t + a_{t+1} Lambda_{t+1}
 *   dC_t[n] += sum_p dy_t[p] S_t[p,n];   dB_t[n] += dt_t sum_p Lambda_t[p,n] x_t[p]
 *   dx_t[p]  = dt_t sum_n Lambda_t[p,n] B_t[n]
 *   ddt_t   += sum_{p,n} Lambda_t[p,n] (A_h a_t S_{t-1}[p,n] + B_t[n] x_t[p])
 *   dA_h    += sum_{t,p,n} Lambda_t[p,n] dt_t a_t S_{t-1}[p,n];   dh0 = a_0 Lambda_0
 * Serial over rows (dB, dC, ddt, dA are sums over several rows), for small
 * problems.  Arguments as oracle_ssd_recurrence plus dy (like x) and dfinal
 * (like h0) in; out: dx (like x), ddt (like dt), dA (nheads), dB, dC (like
 * Bm) and dh0 (like h0, may be NULL).
 */
void oracle_ssd_bwd(const double* x, const double* dt, const double* A_head,
                    const double* Bm, const double* Cm, const double* h0,
                    const double* dy, const double* dfinal,
                    double* dx, double* ddt, double* dA, double* dB, double* dC, double* dh0,
                    int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const size_t nbc = (size_t)batch * seqlen * ngroups * dstate;
    memset(ddt, 0, sizeof(double) * (size_t)batch * seqlen * nheads);
    memset(dA, 0, sizeof(double) * (size_t)nheads);
    memset(dB, 0, sizeof(double) * nbc);
    memset(dC, 0, sizeof(double) * nbc);
    /* Sx[t * dstate + n] is the state entering step t; Sx[(t + 1) * dstate + n] after it */
    double* Sx = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * dstate);
    double* adj = (double*)malloc(sizeof(double) * (size_t)dstate);
    const long long rows = (long long)batch * nheads * headdim;
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        for (int n = 0; n < dstate; ++n) Sx[n] = h0 ? h0[row * dstate + n] : 0.0;
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double step_dt = dt[bt * nheads + h];
            const double decay = exp(A_head[h] * step_dt);
            const double xin = x[(bt * nheads + h) * headdim + p];
            const double* Bt = Bm + (bt * ngroups + g) * dstate;
            for (int n = 0; n < dstate; ++n)
                Sx[(size_t)(t + 1) * dstate + n] =
                    decay * Sx[(size_t)t * dstate + n] + step_dt * xin * Bt[n];
        }
        for (int n = 0; n < dstate; ++n) adj[n] = dfinal ? dfinal[row * dstate + n] : 0.0;
        for (int t = seqlen - 1; t >= 0; --t) {
            const size_t bt = (size_t)b * seqlen + t;
            const size_t ix = (bt * nheads + h) * headdim + p;
            const double step_dt = dt[bt * nheads + h];
            const double decay = exp(A_head[h] * step_dt);
            const double xin = x[ix], dyv = dy[ix];
            const double* Bt = Bm + (bt * ngroups + g) * dstate;
            const double* Ct = Cm + (bt * ngroups + g) * dstate;
            double* dBt = dB + (bt * ngroups + g) * dstate;
            double* dCt = dC + (bt * ngroups + g) * dstate;
            double sum_b = 0.0, sum_dt = 0.0;
            for (int n = 0; n < dstate; ++n) {
                const double s_prev = Sx[(size_t)t * dstate + n];
                adj[n] += dyv * Ct[n];
                dCt[n] += dyv * Sx[(size_t)(t + 1) * dstate + n];
                dBt[n] += adj[n] * step_dt * xin;
                sum_b += adj[n] * Bt[n];
                sum_dt += adj[n] * (A_head[h] * decay * s_prev + Bt[n] * xin);
                dA[h] += adj[n] * step_dt * decay * s_prev;
                adj[n] *= decay;
            }
            dx[ix] = step_dt * sum_b;
            ddt[bt * nheads + h] += sum_dt;
        }
        if (dh0)
            for (int n = 0; n < dstate; ++n) dh0[row * dstate + n] = adj[n];
    }
    free(Sx);
    free(adj);
}

/*
 * Gradient of oracle_mamba3_recurrence for the loss  sum dy . y + sum dfinal .
 * final_state, by differentiating Eq. 9 in reverse.  With Lambda_t = dL/dS_t:
 *   Lambda_t = dy_t (outer) C_t + alpha_{t+1} Lambda_{t+1}
 *   dC_t    += dy_t S_t
 *   x_t and B_t enter twice: with gamma_t at step t and with beta_{t+1} at step t + 1:
 *   dx_t     = gamma_t Lambda_t . B_t + beta_{t+1} Lambda_{t+1} . B_t
 *   dB_t    += (gamma_t Lambda_t + beta_{t+1} Lambda_{t+1}) x_t
 *   d gamma_t = x_t Lambda_t . B_t,  d beta_t = x_{t-1} Lambda_t . B_{t-1},
 *   d alpha_t = Lambda_t . S_{t-1}
 * then through alpha = exp(dt A), gamma = lambda dt, beta = dt (1 - lambda) alpha
 * to ddt, dlambda and dA.  The token before the first (prev_B, prev_x) takes
 * the t = 0 beta term's gradient; dh0 = alpha_0 Lambda_0.  Serial over rows.
 * Arguments as oracle_mamba3_recurrence plus dy, dfinal in; out: dx, ddt,
 * dlam, dA (nheads), dB, dC, dh0 (may be NULL), dprev_B, dprev_x (NULL when
 * prev_B is).
 */
void oracle_mamba3_bwd(const double* x, const double* dt, const double* lam,
                       const double* A_head, const double* Bm, const double* Cm,
                       const double* h0, const double* prev_B, const double* prev_x,
                       const double* dy, const double* dfinal,
                       double* dx, double* ddt, double* dlam, double* dA, double* dB,
                       double* dC, double* dh0, double* dprev_B, double* dprev_x,
                       int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const size_t nbc = (size_t)batch * seqlen * ngroups * dstate;
    memset(ddt, 0, sizeof(double) * (size_t)batch * seqlen * nheads);
    memset(dlam, 0, sizeof(double) * (size_t)batch * seqlen * nheads);
    memset(dA, 0, sizeof(double) * (size_t)nheads);
    memset(dB, 0, sizeof(double) * nbc);
    memset(dC, 0, sizeof(double) * nbc);
    if (dprev_B) memset(dprev_B, 0, sizeof(double) * (size_t)batch * ngroups * dstate);
    double* St = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * dstate);  /* S_{t-1} at t */
    double* adj = (double*)malloc(sizeof(double) * (size_t)dstate);      /* Lambda_t */
    double* carry = (double*)malloc(sizeof(double) * (size_t)dstate);    /* alpha_{t+1} Lambda_{t+1} */
    double* later = (double*)malloc(sizeof(double) * (size_t)dstate);    /* Lambda_{t+1} */
    const long long rows = (long long)batch * nheads * headdim;
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        const double* pB = prev_B ? prev_B + ((size_t)b * ngroups + g) * dstate : NULL;
        const double px = prev_x ? prev_x[row] : 0.0;
        /* forward, every state kept */
        for (int n = 0; n < dstate; ++n) St[n] = h0 ? h0[row * dstate + n] : 0.0;
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double step = dt[bt * nheads + h];
            const double decay = exp(A_head[h] * step);
            const double gam = lam[bt * nheads + h] * step;
            const double bet = (step - gam) * decay;
            const double xin = x[(bt * nheads + h) * headdim + p];
            const double xlast = t > 0 ? x[((bt - 1) * nheads + h) * headdim + p] : px;
            const double* Bcur = Bm + (bt * ngroups + g) * dstate;
            const double* Blast = t > 0 ? Bm + ((bt - 1) * ngroups + g) * dstate : pB;
            for (int n = 0; n < dstate; ++n)
                St[(size_t)(t + 1) * dstate + n] = decay * St[(size_t)t * dstate + n] +
                                                   bet * (Blast ? Blast[n] : 0.0) * xlast +
                                                   gam * Bcur[n] * xin;
        }
        /* reverse */
        for (int n = 0; n < dstate; ++n) {
            carry[n] = dfinal ? dfinal[row * dstate + n] : 0.0;
            later[n] = 0.0;
        }
        double bet_next = 0.0;  /* beta_{t+1} (none past the last step) */
        for (int t = seqlen - 1; t >= 0; --t) {
            const size_t bt = (size_t)b * seqlen + t;
            const size_t ix = (bt * nheads + h) * headdim + p;
            const double step = dt[bt * nheads + h];
            const double lv = lam[bt * nheads + h];
            const double decay = exp(A_head[h] * step);
            const double gam = lv * step;
            const double bet = (step - gam) * decay;
            const double xin = x[ix], dyv = dy[ix];
            const double xlast = t > 0 ? x[((bt - 1) * nheads + h) * headdim + p] : px;
            const double* Bcur = Bm + (bt * ngroups + g) * dstate;
            const double* Blast = t > 0 ? Bm + ((bt - 1) * ngroups + g) * dstate : pB;
            const double* Ccur = Cm + (bt * ngroups + g) * dstate;
            double* dBcur = dB + (bt * ngroups + g) * dstate;
            double* dCcur = dC + (bt * ngroups + g) * dstate;
            double on_B = 0.0, later_on_B = 0.0, on_Blast = 0.0, on_S = 0.0;
            for (int n = 0; n < dstate; ++n) {
                adj[n] = dyv * Ccur[n] + carry[n];
                dCcur[n] += dyv * St[(size_t)(t + 1) * dstate + n];
                on_B += adj[n] * Bcur[n];
                later_on_B += later[n] * Bcur[n];
                if (Blast) on_Blast += adj[n] * Blast[n];
                on_S += adj[n] * St[(size_t)t * dstate + n];
                dBcur[n] += (gam * adj[n] + bet_next * later[n]) * xin;
            }
            dx[ix] = gam * on_B + bet_next * later_on_B;
            const double d_gam = xin * on_B;
            const double d_bet = xlast * on_Blast;
            const double d_alpha = on_S;
            ddt[bt * nheads + h] += d_gam * lv +
                                    d_bet * ((1.0 - lv) * decay + step * (1.0 - lv) * A_head[h] * decay) +
                                    d_alpha * A_head[h] * decay;
            dlam[bt * nheads + h] += d_gam * step - d_bet * step * decay;
            dA[h] += d_bet * step * (1.0 - lv) * step * decay + d_alpha * step * decay;
            if (t == 0 && pB) {
                if (dprev_x) dprev_x[row] = bet * on_Blast;
                if (dprev_B)
                    for (int n = 0; n < dstate; ++n)
                        dprev_B[((size_t)b * ngroups + g) * dstate + n] += bet * adj[n] * px;
            }
            for (int n = 0; n < dstate; ++n) {
                later[n] = adj[n];
                carry[n] = decay * adj[n];
            }
            bet_next = bet;
        }
        if (dh0)
            for (int n = 0; n < dstate; ++n) dh0[row * dstate + n] = carry[n];
        if (dprev_x && seqlen == 0) dprev_x[row] = 0.0;
    }
    free(St);
    free(adj);
    free(carry);
    free(later);
}

/*
 * Gradient of oracle_mamba3_mimo_recurrence for the loss  sum dy . y + sum
 * dfinal . final_state, by differentiating the rank-R recurrence in reverse.
 * Per row (b, h, p) with bx_t[n] = sum_r B_t[n,r] x_t[p,r] and Lambda_t = dL/dS_t:
 *   Lambda_t  = sum_r dy_t[p,r] C_t[:,r] + alpha_{t+1} Lambda_{t+1}
 *   dC_t[:,r] += dy_t[p,r] S_t
 *   bx_t enters with gamma_t at step t and with beta_{t+1} at step t + 1, so
 *   d bx_t = gamma_t Lambda_t + beta_{t+1} Lambda_{t+1}, and
 *   dx_t[p,r] = d bx_t . B_t[:,r],  dB_t[:,r] += d bx_t x_t[p,r];
 *   d gamma_t = Lambda_t . bx_t,  d beta_t = Lambda_t . bx_{t-1},  d alpha_t = Lambda_t . S_{t-1}
 * then through alpha, gamma, beta to ddt, dlambda and dA as in
 * oracle_mamba3_bwd.  The token before the first takes the t = 0 beta term's
 * gradient; dh0 = alpha_0 Lambda_0.  Serial over rows.  Arguments as
 * oracle_mamba3_mimo_recurrence plus dy (like x), dfinal in; out: dx (like
 * x), ddt, dlam, dA (nheads), dB, dC (like B), dh0 (may be NULL), dprev_B,
 * dprev_x (like prev_B, prev_x; NULL when prev_B is).
 */
void oracle_mamba3_mimo_bwd(const double* x, const double* dt, const double* lam,
                            const double* A_head, const double* Bm, const double* Cm,
                            const double* h0, const double* prev_B, const double* prev_x,
                            const double* dy, const double* dfinal,
                            double* dx, double* ddt, double* dlam, double* dA, double* dB,
                            double* dC, double* dh0, double* dprev_B, double* dprev_x,
                            int batch, int seqlen, int rank, int nheads, int headdim, int dstate,
                            int ngroups)
{
    const int heads_per_group = nheads / ngroups;
    const size_t nbc = (size_t)batch * seqlen * rank * ngroups * dstate;
    memset(ddt, 0, sizeof(double) * (size_t)batch * seqlen * nheads);
    memset(dlam, 0, sizeof(double) * (size_t)batch * seqlen * nheads);
    memset(dA, 0, sizeof(double) * (size_t)nheads);
    memset(dB, 0, sizeof(double) * nbc);
    memset(dC, 0, sizeof(double) * nbc);
    if (dprev_B) memset(dprev_B, 0, sizeof(double) * (size_t)batch * rank * ngroups * dstate);
    if (dprev_x) memset(dprev_x, 0, sizeof(double) * (size_t)batch * rank * nheads * headdim);
    const size_t ns = (size_t)dstate;
    double* St = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * ns);  /* S_{t-1} at t */
    double* BX = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * ns);  /* bx_{t-1} at t */
    double* adj = (double*)malloc(sizeof(double) * ns);    /* Lambda_t */
    double* carry = (double*)malloc(sizeof(double) * ns);  /* alpha_{t+1} Lambda_{t+1} */
    double* later = (double*)malloc(sizeof(double) * ns);  /* Lambda_{t+1} */
    double* dbx = (double*)malloc(sizeof(double) * ns);
    const long long rows = (long long)batch * nheads * headdim;
    for (long long row = 0; row < rows; ++row) {
        const int p = (int)(row % headdim);
        const int h = (int)((row / headdim) % nheads);
        const int b = (int)(row / ((long long)headdim * nheads));
        const int g = h / heads_per_group;
        const int has_prev = prev_B && prev_x;
#define XI(bt, r) ((((size_t)(bt) * rank + (r)) * nheads + h) * headdim + p)
#define BI(bt, r) ((((size_t)(bt) * rank + (r)) * ngroups + g) * ns)
        /* forward, every state and every bx kept */
        for (size_t n = 0; n < ns; ++n) {
            St[n] = h0 ? h0[row * dstate + n] : 0.0;
            double bx = 0.0;
            if (has_prev)
                for (int r = 0; r < rank; ++r)
                    bx += prev_B[(((size_t)b * rank + r) * ngroups + g) * ns + n] *
                          prev_x[(((size_t)b * rank + r) * nheads + h) * headdim + p];
            BX[n] = bx;
        }
        for (int t = 0; t < seqlen; ++t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double step = dt[bt * nheads + h];
            const double decay = exp(A_head[h] * step);
            const double gam = lam[bt * nheads + h] * step;
            const double bet = (step - gam) * decay;
            for (size_t n = 0; n < ns; ++n) {
                double bx = 0.0;
                for (int r = 0; r < rank; ++r) bx += Bm[BI(bt, r) + n] * x[XI(bt, r)];
                BX[(size_t)(t + 1) * ns + n] = bx;
                St[(size_t)(t + 1) * ns + n] = decay * St[(size_t)t * ns + n] +
                                               bet * BX[(size_t)t * ns + n] + gam * bx;
            }
        }
        /* reverse */
        for (size_t n = 0; n < ns; ++n) {
            carry[n] = dfinal ? dfinal[row * dstate + n] : 0.0;
            later[n] = 0.0;
        }
        double bet_next = 0.0;  /* beta_{t+1} (none past the last step) */
        double bet0 = 0.0;
        for (int t = seqlen - 1; t >= 0; --t) {
            const size_t bt = (size_t)b * seqlen + t;
            const double step = dt[bt * nheads + h];
            const double lv = lam[bt * nheads + h];
            const double decay = exp(A_head[h] * step);
            const double gam = lv * step;
            const double bet = (step - gam) * decay;
            double on_bx = 0.0, on_bxlast = 0.0, on_S = 0.0;
            for (size_t n = 0; n < ns; ++n) {
                double a = carry[n];
                for (int r = 0; r < rank; ++r) {
                    const double dyv = dy[XI(bt, r)];
                    a += dyv * Cm[BI(bt, r) + n];
                    dC[BI(bt, r) + n] += dyv * St[(size_t)(t + 1) * ns + n];
                }
                adj[n] = a;
                on_bx += a * BX[(size_t)(t + 1) * ns + n];
                on_bxlast += a * BX[(size_t)t * ns + n];
                on_S += a * St[(size_t)t * ns + n];
                dbx[n] = gam * a + bet_next * later[n];
            }
            for (int r = 0; r < rank; ++r) {
                double acc = 0.0;
                const double xv = x[XI(bt, r)];
                for (size_t n = 0; n < ns; ++n) {
                    acc += dbx[n] * Bm[BI(bt, r) + n];
                    dB[BI(bt, r) + n] += dbx[n] * xv;
                }
                dx[XI(bt, r)] = acc;
            }
            const double d_gam = on_bx, d_bet = on_bxlast, d_alpha = on_S;
            ddt[bt * nheads + h] += d_gam * lv +
                                    d_bet * ((1.0 - lv) * decay + step * (1.0 - lv) * A_head[h] * decay) +
                                    d_alpha * A_head[h] * decay;
            dlam[bt * nheads + h] += step * (d_gam - d_bet * decay);
            dA[h] += d_bet * step * (1.0 - lv) * step * decay + d_alpha * step * decay;
            for (size_t n = 0; n < ns; ++n) {
                later[n] = adj[n];
                carry[n] = adj[n] * decay;
            }
            bet_next = bet;
            bet0 = bet;
        }
        if (has_prev && seqlen > 0 && dprev_B && dprev_x) {
            /* bx_{-1} entered with beta_0 at step 0: d bx_{-1} = beta_0 Lambda_0 (= later) */
            for (int r = 0; r < rank; ++r) {
                const double* pBr = prev_B + (((size_t)b * rank + r) * ngroups + g) * ns;
                const size_t ixr = (((size_t)b * rank + r) * nheads + h) * headdim + p;
                double acc = 0.0;
                for (size_t n = 0; n < ns; ++n) {
                    acc += bet0 * later[n] * pBr[n];
                    dprev_B[(((size_t)b * rank + r) * ngroups + g) * ns + n] +=
                        bet0 * later[n] * prev_x[ixr];
                }
                dprev_x[ixr] = acc;
            }
        }
        if (dh0)
            for (size_t n = 0; n < ns; ++n) dh0[row * dstate + n] = carry[n];
#undef XI
#undef BI
    }
    free(St);
    free(BX);
    free(adj);
    free(carry);
    free(later);
    free(dbx);
}

/*
 * oracle_mamba3_rope -- [P2] "How it works", Phase 1: the angle cumsum
 * cum_angles = -cumsum(dt * theta) along the sequence, then RoPE applied to
 * B and C.  Readings taken where the page is silent:
 *  - theta holds one angular rate per (batch, step, head, state pair), so it
 *    multiplies dt elementwise; the heads of a group rotate the group's B
 *    and C by their own angles, so the results have one row per head.
 *  - State pair k is (2k, 2k + 1), rotated as the complex number
 *    B[2k] + i B[2k+1] times exp(i angle) (the original RoPE pairing).
 *  - The cumsum is inclusive: step t's angle includes dt_t theta_t.  The
 *    angle entering the sequence is angle0 (0 when NULL); the angle after the
 *    last step is written to angle_out (when not NULL), so a resumed prefill
 *    or a decode step continues the sequence.
 *  - MIMO: every rank of a step is rotated by the step's angle.
 * Layouts: B, C [batch][L][R][G][N]; dt [batch][L][H]; theta, the angles
 * [batch][L][H][N/2] and [batch][H][N/2]; Brot, Crot [batch][L][R][H][N].
 */
void oracle_mamba3_rope(const double* Bm, const double* Cm, const double* dt,
                        const double* theta, const double* angle0, double* Brot, double* Crot,
                        double* angle_out, int batch, int seqlen, int rank, int nheads,
                        int ngroups, int dstate)
{
    const int half = dstate / 2;
    const int heads_per_group = nheads / ngroups;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < nheads; ++h) {
            const int g = h / heads_per_group;
            for (int k = 0; k < half; ++k) {
                const size_t ai = ((size_t)b * nheads + h) * half + k;
                double angle = angle0 ? angle0[ai] : 0.0;
                for (int t = 0; t < seqlen; ++t) {
                    const size_t bt = (size_t)b * seqlen + t;
                    angle -= dt[bt * nheads + h] * theta[(bt * nheads + h) * half + k];
                    const double c = cos(angle), sn = sin(angle);
                    for (int r = 0; r < rank; ++r) {
                        const size_t src = ((bt * rank + r) * ngroups + g) * dstate + 2 * k;
                        const size_t dst = ((bt * rank + r) * nheads + h) * dstate + 2 * k;
                        Brot[dst] = Bm[src] * c - Bm[src + 1] * sn;
                        Brot[dst + 1] = Bm[src] * sn + Bm[src + 1] * c;
                        Crot[dst] = Cm[src] * c - Cm[src + 1] * sn;
                        Crot[dst + 1] = Cm[src] * sn + Cm[src + 1] * c;
                    }
                }
                if (angle_out) angle_out[ai] = angle;
            }
        }
    }
}

int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
