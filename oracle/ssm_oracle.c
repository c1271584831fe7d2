/*
 * ssm_oracle.c -- fp64 CPU oracle for the selective-scan forward and the
 * single-token state update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (plain definition, no blocking, fusion or reordering):
 *
 *   for every batch row b and channel d, with h[n] = h0[b,d,n] (or 0):
 *     for l = 0 .. L-1:
 *       x     = delta[b,d,l] + bias[d]
 *       dt    = softplus(x)  (or x when softplus is off)
 *       for n:
 *         Abar  = exp(dt * A[d,n])
 *         coef  = (exp(dt*A) - 1) / A[d,n]      (coef = dt when A[d,n] == 0)
 *                 (coef = dt for every n with the Euler input term, `euler`)
 *         h[n]  = Abar * h[n] + coef * B[b,n,l] * u[b,d,l]
 *       y     = sum_n C[b,n,l] * h[n] + D[d] * u[b,d,l]
 *       y    *= silu(z[b,d,l])                  (when z is given)
 *     h_last[b,d,:] = h
 *
 * Passages followed:
 *  - zero-order-hold discretisation Abar = exp(dA), Bbar = (dA)^-1 (exp(dA) - I) dB:
 *    velog review of "Mamba: Linear-Time Sequence Modeling with Selective
 *    State Spaces", section 2 "Discretization"; the derivation and the
 *    invertibility condition on A are in "mamba 学习" (fakeeyes2wo), section
 *    "MAMBA" (integral of e^{A tau} = A^-1 (e^{A dt} - I)).  For diagonal A the
 *    matrix expression is elementwise, giving coef above; its A -> 0 limit is dt.
 *  - recurrence h_k = Abar h_{k-1} + Bbar x_k, y_k = C h_k (inclusive
 *    convention): velog review, section 2 "Discretization", item 3.
 *  - D skip y += D x: "mamba 学习", section "SSM 状态空间模型" (output equation)
 *    and Mamba_Model_Report.md section 4.2 (y = y + D * x).
 *  - gate y * silu(z), applied after the D skip: Mamba_Model_Report.md section 3
 *    (MambaBlock.forward: z = silu(z); output = y * z).
 *  - dt = softplus(raw + bias): "Mamba学习记录" (lengnian), section "怎么增加选择性"
 *    (tau_delta = softplus) and velog review section 3.2 (broadcast, add the
 *    parameter, softplus).
 *  - h starts at zero: Mamba_Model_Report.md section 4.2 (selective_scan_seq
 *    starts from torch.zeros) and "mamba 学习" (h_0 = 0).
 *  - decode step: Mamba_Model_Report.md section 6 (ssm_step: h = deltaA * h + BX;
 *    y = h @ C + D * x), with the same discretisation.
 *  - Euler input term Bbar = dt * B (selected by `euler`): Mamba_Model_Report.md
 *    section 4.2 (selective_scan: deltaB = delta * B, BX = deltaB * x), with the
 *    same Abar = exp(dt * A).
 *
 * The file also holds the scan's gradient (oracle_scan_bwd, the reverse-mode
 * derivative of the loop above, written out below) and the causal depthwise
 * convolution that precedes the scan in the report's MambaBlock
 * (oracle_conv1d_fwd, oracle_conv1d_update; definitions and passages at the end).
 *
 * Pinned by tests/test_oracle_pins.py against brute-force unrolled sums,
 * the LTI convolution form, a geometric-series closed form, the A -> 0 limit,
 * linearity in u, step/scan equivalence and split invariance.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), in a form that neither overflows nor loses
 * the small-x tail. */
static double oracle_softplus(double x)
{
    if (x > 0.0)
        return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^{-z}) */
static double oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* One recurrence step for channel (b, d) at one position.
 * h has dstate entries; B_col/C_col are the dstate values of B and C at this
 * position, read with stride `bc_stride` between consecutive n. */
static double oracle_step(int64_t dstate, double* h, double u, double delta_raw,
                          double bias, int delta_softplus, const double* A_row,
                          const double* B_col, const double* C_col, int64_t bc_stride,
                          double Dd, const double* z, int euler)
{
    double x = delta_raw + bias;
    double dt = delta_softplus ? oracle_softplus(x) : x;
    double acc = 0.0;
    for (int64_t n = 0; n < dstate; ++n) {
        double a = A_row[n];
        double Abar = exp(dt * a);
        double coef = (a == 0.0) ? dt : expm1(dt * a) / a;
        if (euler)
            coef = dt;
        h[n] = Abar * h[n] + coef * B_col[n * bc_stride] * u;
        acc += C_col[n * bc_stride] * h[n];
    }
    double y = acc + Dd * u;
    if (z)
        y *= oracle_silu(*z);
    return y;
}

/* Scan one (b, d) row over all L positions. */
static void oracle_scan_row(int64_t b, int64_t d, int64_t dim, int64_t dstate, int64_t seqlen,
                            const double* u, const double* delta, const double* delta_bias,
                            int delta_softplus, const double* A, const double* B,
                            const double* C, const double* D, const double* z,
                            const double* h0, double* h_last, double* y, double* h, int euler)
{
    const int64_t row = b * dim + d;
    for (int64_t n = 0; n < dstate; ++n)
        h[n] = h0 ? h0[row * dstate + n] : 0.0;
    const double bias = delta_bias ? delta_bias[d] : 0.0;
    const double Dd = D ? D[d] : 0.0;
    for (int64_t l = 0; l < seqlen; ++l) {
        const int64_t i = row * seqlen + l;
        const double* Bcol = B + b * dstate * seqlen + l;
        const double* Ccol = C + b * dstate * seqlen + l;
        y[i] = oracle_step(dstate, h, u[i], delta[i], bias, delta_softplus, A + d * dstate,
                           Bcol, Ccol, seqlen, Dd, z ? z + i : NULL, euler);
    }
    if (h_last)
        for (int64_t n = 0; n < dstate; ++n)
            h_last[row * dstate + n] = h[n];
}

/* Full scan.  Rows are independent; `nthreads` > 1 only spreads whole rows
 * over threads and does not change any arithmetic.
 * Returns 0 on success, -1 on bad sizes or allocation failure. */
int oracle_scan_fwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                    const double* u, const double* delta, const double* delta_bias,
                    int delta_softplus, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* h0, double* h_last,
                    double* y, int nthreads, int euler)
{
    if (batch < 0 || dim < 0 || dstate <= 0 || seqlen < 0)
        return -1;
    const int64_t rows = batch * dim;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
        if (!h) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < rows; ++r)
                oracle_scan_row(r / dim, r % dim, dim, dstate, seqlen, u, delta, delta_bias,
                                delta_softplus, A, B, C, D, z, h0, h_last, y, h, euler);
            free(h);
        }
    }
    (void)nthreads;
    return failed ? -1 : 0;
}

/* Scan only the listed rows (row = b * dim + d).  y_rows is [nrows, seqlen],
 * h_last_rows (optional) is [nrows, dstate], h0 (optional) is the full
 * [batch, dim, dstate] tensor.  Used for sampled parity at full sizes. */
int oracle_scan_rows(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                     const int64_t* rows, int64_t nrows,
                     const double* u_rows, const double* delta_rows, const double* delta_bias,
                     int delta_softplus, const double* A, const double* B, const double* C,
                     const double* D, const double* z_rows, const double* h0,
                     double* h_last_rows, double* y_rows, int euler)
{
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || nrows < 0)
        return -1;
    double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
    if (!h)
        return -1;
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t r = rows[k];
        if (r < 0 || r >= batch * dim) {
            free(h);
            return -1;
        }
        const int64_t b = r / dim, d = r % dim;
        for (int64_t n = 0; n < dstate; ++n)
            h[n] = h0 ? h0[r * dstate + n] : 0.0;
        const double bias = delta_bias ? delta_bias[d] : 0.0;
        const double Dd = D ? D[d] : 0.0;
        for (int64_t l = 0; l < seqlen; ++l) {
            const int64_t i = k * seqlen + l;
            y_rows[i] = oracle_step(dstate, h, u_rows[i], delta_rows[i], bias, delta_softplus,
                                    A + d * dstate, B + b * dstate * seqlen + l,
                                    C + b * dstate * seqlen + l, seqlen, Dd,
                                    z_rows ? z_rows + i : NULL, euler);
        }
        if (h_last_rows)
            for (int64_t n = 0; n < dstate; ++n)
                h_last_rows[k * dstate + n] = h[n];
    }
    free(h);
    return 0;
}

/* Single-token state update, h updated in place.
 * h [batch, dim, dstate]; u, delta, z, y [batch, dim]; B, C [batch, dstate].
 * Channels are independent; `nthreads` > 1 only spreads whole channels over
 * threads and does not change any arithmetic. */
int oracle_state_update(int64_t batch, int64_t dim, int64_t dstate, double* h,
                        const double* u, const double* delta, const double* delta_bias,
                        int delta_softplus, const double* A, const double* B, const double* C,
                        const double* D, const double* z, double* y, int euler, int nthreads)
{
    if (batch < 0 || dim < 0 || dstate <= 0)
        return -1;
    const int64_t rows = batch * dim;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t b = i / dim, d = i % dim;
        y[i] = oracle_step(dstate, h + i * dstate, u[i], delta[i],
                           delta_bias ? delta_bias[d] : 0.0, delta_softplus,
                           A + d * dstate, B + b * dstate, C + b * dstate, 1,
                           D ? D[d] : 0.0, z ? z + i : NULL, euler);
    }
    (void)nthreads;
    return 0;
}

/* ------------------------------------------------------------------------
 * Causal depthwise convolution over time (the step before the scan).
 *
 *   out[b,d,l] = act( bias[d] + sum_{k=0}^{W-1} w[d,k] * x[b,d,l-(W-1)+k] )
 *
 * where x at a position before 0 is the carried-in window state_in[b,d,(W-1)+p]
 * (zero without a state), and act is silu or the identity.  This is the
 * MambaBlock's nn.Conv1d(groups=d_inner, kernel_size=d_conv, padding=d_conv-1)
 * truncated to the first L outputs, followed by silu (Mamba_Model_Report.md
 * section 3, MambaBlock.forward: x = self.conv1d(x)[:, :, :L]; x = F.silu(x)).
 * state_out[b,d,j] (optional) receives the last W-1 inputs, positions
 * L-(W-1)+j, which is the decode cache the report keeps (section 6: inputs,
 * (B, ED, d_conv-1)).
 * ------------------------------------------------------------------------ */
static double oracle_conv_input(const double* x_row, const double* state_row, int64_t width,
                                int64_t p)
{
    if (p >= 0)
        return x_row[p];
    if (p < -(width - 1) || !state_row)
        return 0.0;
    return state_row[(width - 1) + p];
}

int oracle_conv1d_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                      const double* x, const double* weight, const double* bias,
                      const double* state_in, int apply_silu, double* out, double* state_out)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t row = b * dim + d;
            const double* xr = x + row * seqlen;
            const double* sr = state_in ? state_in + row * (width - 1) : NULL;
            for (int64_t l = 0; l < seqlen; ++l) {
                double acc = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < width; ++k)
                    acc += weight[d * width + k] * oracle_conv_input(xr, sr, width,
                                                                     l - (width - 1) + k);
                out[row * seqlen + l] = apply_silu ? oracle_silu(acc) : acc;
            }
            if (state_out)
                for (int64_t j = 0; j < width - 1; ++j)
                    state_out[row * (width - 1) + j] =
                        oracle_conv_input(xr, sr, width, seqlen - (width - 1) + j);
        }
    }
    return 0;
}

/* One decode position (Mamba_Model_Report.md section 6, step): the window is the
 * cached W-1 inputs followed by x; out = act(bias + sum_k w[k] window[k]); the
 * cache drops its oldest input and appends x.  state [b,d,W-1] is updated in place. */
int oracle_conv1d_update(int64_t batch, int64_t dim, int64_t width, double* state,
                         const double* x, const double* weight, const double* bias,
                         int apply_silu, double* out)
{
    if (batch < 0 || dim < 0 || width < 1)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t row = b * dim + d;
            double* s = state + row * (width - 1);
            double acc = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < width - 1; ++k)
                acc += weight[d * width + k] * s[k];
            acc += weight[d * width + width - 1] * x[row];
            out[row] = apply_silu ? oracle_silu(acc) : acc;
            for (int64_t k = 0; k + 1 < width - 1; ++k)
                s[k] = s[k + 1];
            if (width > 1)
                s[width - 2] = x[row];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Gradient of the scan (reverse mode), for training.  Mamba_Model_Report.md
 * section 4.1 gives the recurrence H[t] = A[t] H[t-1] + X[t] a backward pass
 * built from a reverse scan (pscan_rev) that yields the gradients of A and X;
 * "Mamba学习记录" (lengnian), Part3, lists recomputation of intermediate
 * results among the hardware-aware algorithm's means.  The oracle is the chain
 * rule applied to the loop of oracle_step, one position at a time in reverse,
 * with every forward state kept (no recomputation needed at oracle sizes):
 *
 *   given dy[b,d,l] (and optionally dh_last[b,d,n]), with the forward states
 *   h_l (h_{-1} = h0) of the channel kept in full:
 *     g[n] = dh_last[n] (or 0)                        g = dLoss/dh_l
 *     for l = L-1 .. 0:
 *       y0   = sum_n C[n,l] h_l[n] + D u_l            (output before the gate)
 *       dz_l = dy_l * y0 * silu'(z_l);  dy0 = dy_l * silu(z_l)   (no z: dy0 = dy_l)
 *       dD  += dy0 u_l;  du_l = D dy0
 *       for n:
 *         g[n]      += C[n,l] dy0                     (y0 depends on h_l)
 *         dC[n,l]   += dy0 h_l[n]                     (summed over the channels d)
 *         h_l = Abar h_{l-1} + coef B u, so with p = g[n] h_{l-1}[n], r = g[n] B u:
 *         dB[n,l]   += g[n] coef u                    (summed over d)
 *         du_l      += g[n] coef B[n,l]
 *         ddt       += p * dAbar/ddt + r * dcoef/ddt
 *         dA[d,n]   += p * dAbar/da  + r * dcoef/da   (summed over b, l)
 *         g[n]       = Abar g[n]                      (dLoss/dh_{l-1})
 *       dx = ddt * softplus'(x) (= ddt * sigmoid(x); ddt without softplus)
 *       ddelta_l = dx;  dbias[d] += dx
 *     dh0 = g
 *
 * with Abar = exp(dt a): dAbar/ddt = a Abar, dAbar/da = dt Abar; and
 * ZOH coef = expm1(dt a)/a: dcoef/ddt = Abar, dcoef/da = (dt Abar - coef)/a
 * (at a == 0: coef = dt, dcoef/ddt = 1, dcoef/da = dt^2/2, the limit); Euler
 * coef = dt: dcoef/ddt = 1, dcoef/da = 0.  For 0 < |dt a| < 1e-3, dcoef/da is
 * taken from its Taylor series dt^2 (1/2 + q/3 + q^2/8 + q^3/30) (q = dt a;
 * the first dropped term, q^4/144, is below 1e-14 of the sum) because the
 * difference above cancels there.
 * silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))).
 *
 * Pinned by tests/pins.py: central finite differences of the forward oracle
 * on every input, and the exact identities of a function linear in (u, h0),
 * in B and in C.
 * ------------------------------------------------------------------------ */
static double oracle_sigmoid(double x)
{
    return 1.0 / (1.0 + exp(-x));
}

/* dcoef/da of the ZOH input coefficient coef = expm1(dt a)/a */
static double oracle_dcoef_da(double dt, double a, double Abar, double coef)
{
    if (a == 0.0)
        return 0.5 * dt * dt;
    const double q = dt * a;
    if (fabs(q) < 1e-3)
        return dt * dt * (0.5 + q * (1.0 / 3.0 + q * (1.0 / 8.0 + q * (1.0 / 30.0))));
    return (dt * Abar - coef) / a;
}

/* Backward of one channel (b, d).  hs is scratch of (L + 1) * dstate doubles;
 * dB_acc, dC_acc ([batch, dstate, L]), dA_acc ([dim, dstate]), dD_acc, dbias_acc
 * ([dim]) are accumulated into; du, ddelta, dz, dh0 are written for this row. */
static void oracle_bwd_row(int64_t b, int64_t d, int64_t dim, int64_t dstate, int64_t seqlen,
                           const double* u, const double* delta, const double* delta_bias,
                           int delta_softplus, const double* A, const double* B,
                           const double* C, const double* D, const double* z,
                           const double* h0, const double* dy, const double* dh_last,
                           double* du, double* ddelta, double* dz, double* dh0,
                           double* dA_acc, double* dB_acc, double* dC_acc, double* dD_acc,
                           double* dbias_acc, double* hs, double* g, int euler)
{
    const int64_t row = b * dim + d;
    const double bias = delta_bias ? delta_bias[d] : 0.0;
    const double Dd = D ? D[d] : 0.0;
    const double* Arow = A + d * dstate;
    const double* Bb = B + b * dstate * seqlen;
    const double* Cb = C + b * dstate * seqlen;

    /* forward, keeping every state: hs[(l + 1) * dstate + n] = h_l[n] */
    for (int64_t n = 0; n < dstate; ++n)
        hs[n] = h0 ? h0[row * dstate + n] : 0.0;
    for (int64_t l = 0; l < seqlen; ++l) {
        const int64_t i = row * seqlen + l;
        const double x = delta[i] + bias;
        const double dt = delta_softplus ? oracle_softplus(x) : x;
        for (int64_t n = 0; n < dstate; ++n) {
            const double a = Arow[n];
            const double Abar = exp(dt * a);
            const double coef = euler ? dt : (a == 0.0 ? dt : expm1(dt * a) / a);
            hs[(l + 1) * dstate + n] = Abar * hs[l * dstate + n] + coef * Bb[n * seqlen + l] * u[i];
        }
    }

    /* reverse */
    for (int64_t n = 0; n < dstate; ++n)
        g[n] = dh_last ? dh_last[row * dstate + n] : 0.0;
    for (int64_t l = seqlen - 1; l >= 0; --l) {
        const int64_t i = row * seqlen + l;
        const double x = delta[i] + bias;
        const double dt = delta_softplus ? oracle_softplus(x) : x;
        const double* h_l = hs + (l + 1) * dstate;
        const double* h_prev = hs + l * dstate;
        double y0 = Dd * u[i];
        for (int64_t n = 0; n < dstate; ++n)
            y0 += Cb[n * seqlen + l] * h_l[n];
        double dy0 = dy[i];
        if (z) {
            const double sg = oracle_sigmoid(z[i]);
            dz[i] = dy[i] * y0 * sg * (1.0 + z[i] * (1.0 - sg));
            dy0 = dy[i] * z[i] * sg;
        }
        dD_acc[d] += dy0 * u[i];
        double du_l = Dd * dy0;
        double ddt = 0.0;
        for (int64_t n = 0; n < dstate; ++n) {
            const double a = Arow[n];
            const double Bv = Bb[n * seqlen + l];
            g[n] += Cb[n * seqlen + l] * dy0;
            dC_acc[b * dstate * seqlen + n * seqlen + l] += dy0 * h_l[n];
            const double Abar = exp(dt * a);
            double coef, dcoef_ddt, dcoef_da;
            if (euler) {
                coef = dt;
                dcoef_ddt = 1.0;
                dcoef_da = 0.0;
            } else if (a == 0.0) {
                coef = dt;
                dcoef_ddt = 1.0;
                dcoef_da = oracle_dcoef_da(dt, a, Abar, coef);
            } else {
                coef = expm1(dt * a) / a;
                dcoef_ddt = Abar;
                dcoef_da = oracle_dcoef_da(dt, a, Abar, coef);
            }
            const double p = g[n] * h_prev[n];
            const double r = g[n] * Bv * u[i];
            dB_acc[b * dstate * seqlen + n * seqlen + l] += g[n] * coef * u[i];
            du_l += g[n] * coef * Bv;
            ddt += p * a * Abar + r * dcoef_ddt;
            dA_acc[d * dstate + n] += p * dt * Abar + r * dcoef_da;
            g[n] = Abar * g[n];
        }
        const double dx = delta_softplus ? ddt * oracle_sigmoid(x) : ddt;
        ddelta[i] = dx;
        dbias_acc[d] += dx;
        du[i] = du_l;
    }
    if (dh0)
        for (int64_t n = 0; n < dstate; ++n)
            dh0[row * dstate + n] = g[n];
}

/* Gradient of the full scan.  Per-row outputs du, ddelta [b,d,l], dz [b,d,l]
 * (when z), dh0 [b,d,n] (optional); reductions dA [d,n], dB, dC [b,n,l], dD,
 * ddelta_bias [d] (each optional except dB, dC, dA).  Rows are spread over
 * `nthreads` threads with private accumulators summed in thread order at the end.
 * Returns 0 on success, -1 on bad sizes or allocation failure. */
int oracle_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                    const double* u, const double* delta, const double* delta_bias,
                    int delta_softplus, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* h0, const double* dy,
                    const double* dh_last, double* du, double* ddelta, double* dA, double* dB,
                    double* dC, double* dD, double* dz, double* ddelta_bias, double* dh0,
                    int nthreads, int euler)
{
    if (batch < 0 || dim < 0 || dstate <= 0 || seqlen < 0)
        return -1;
    const int64_t rows = batch * dim;
    const size_t nbc = (size_t)(batch * dstate * seqlen), na = (size_t)(dim * dstate);
    if (nthreads < 1)
        nthreads = 1;
#ifndef _OPENMP
    nthreads = 1;
#endif
    /* private accumulators: [thread][dA | dB | dC | dD | dbias] */
    const size_t per = na + 2 * nbc + 2 * (size_t)dim;
    double* acc = (double*)calloc(per * (size_t)nthreads, sizeof(double));
    if (!acc)
        return -1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        int t = 0;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        double* mine = acc + per * (size_t)t;
        double* hs = (double*)malloc(sizeof(double) * (size_t)((seqlen + 1) * dstate));
        double* g = (double*)malloc(sizeof(double) * (size_t)dstate);
        if (!hs || !g) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
            for (int64_t r = 0; r < rows; ++r)
                oracle_bwd_row(r / dim, r % dim, dim, dstate, seqlen, u, delta, delta_bias,
                               delta_softplus, A, B, C, D, z, h0, dy, dh_last, du, ddelta, dz,
                               dh0, mine, mine + na, mine + na + nbc, mine + na + 2 * nbc,
                               mine + na + 2 * nbc + dim, hs, g, euler);
        }
        free(hs);
        free(g);
    }
    if (!failed) {
        for (size_t k = 0; k < na; ++k) {
            double s = 0.0;
            for (int t = 0; t < nthreads; ++t)
                s += acc[per * (size_t)t + k];
            dA[k] = s;
        }
        for (size_t k = 0; k < nbc; ++k) {
            double sb = 0.0, sc = 0.0;
            for (int t = 0; t < nthreads; ++t) {
                sb += acc[per * (size_t)t + na + k];
                sc += acc[per * (size_t)t + na + nbc + k];
            }
            dB[k] = sb;
            dC[k] = sc;
        }
        for (int64_t k = 0; k < dim; ++k) {
            double sd = 0.0, sbias = 0.0;
            for (int t = 0; t < nthreads; ++t) {
                sd += acc[per * (size_t)t + na + 2 * nbc + (size_t)k];
                sbias += acc[per * (size_t)t + na + 2 * nbc + (size_t)dim + (size_t)k];
            }
            if (dD)
                dD[k] = sd;
            if (ddelta_bias)
                ddelta_bias[k] = sbias;
        }
    }
    free(acc);
    return failed ? -1 : 0;
}
