/*
 * Selective-scan oracle: a plain, slow, sequential fp64 CPU evaluation of the
 * Mamba selective state-space recurrence and of its single-token decode update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources (the web pages the method is taken from):
 *   [M]  "mamba-metal: Apple Silicon で Mamba を動かす" (createcentury blog #4),
 *        section "Selective scan の本質" (h_t = Ā_t h_{t-1} + B̄_t u_t, y_t = C_tᵀ h_t,
 *        Ā_t = exp(Δ_t A)), section "チャンク間 running prefix" (carry combined from
 *        the left), section "O(L) インクリメンタルデコード" (the per-token update
 *        h_new = exp(Δ A_s) h + Δ x B_s, y = Σ_s h_new C_s + D x, then the z gate).
 *   [K]  the same blog's walkthrough of the official CUDA forward kernel (title lost
 *        in the feed extraction), section "なぜ「scan」か" (the pair a_i = exp(Δ A),
 *        b_i = Δ B u, and the associative operator), section "1チャンク内の処理フロー"
 *        (softplus on Δ, out = D·u, out += h·C per state, out *= z·sigmoid(z)).
 *   [S]  SpeechLens docs/kernel-optimization.md, MetalSelectiveScan section (tensor
 *        contract: A_log [D,N], B,C [B,L,N], delta_raw,u,z [B,L,D], D [D]; the kernel
 *        takes raw A_log and applies -exp(A_log); softplus log(1+exp(x)) on delta_raw).
 *
 * Readings where the pages are silent:
 *   - B̄ is the Euler form b = Δ·B·u ([K] writes the pair's second element as Δ B u).
 *   - delta_bias (per channel, NULL = 0) is added to delta_raw before softplus.
 *   - softplus(x) = max(x,0) + log1p(exp(-|x|)), the exact overflow-free form.
 *   - h_{-1} = 0 unless an initial state h0 is given; the D skip is added before the
 *     gate; silu(z) = z / (1 + exp(-z)).
 *   - h0 (the initial-state input) is the state a previous call left behind: the carry
 *     of [M] "チャンク間 running prefix" handed across calls instead of across chunks, the
 *     prefill state that [M] "O(L) インクリメンタルデコード" continues from.
 *   - B and C are shared by all channels of a batch row: [B,L,N]; last_state is [B,D,N].
 *
 * Layouts (all contiguous, row-major): u, delta_raw, z : [batch, L, Dm];
 * B, C : [batch, L, N]; A_log : [Dm, N]; D, delta_bias : [Dm].
 * Inputs arrive as float (the exact values the GPU path consumes); every
 * arithmetic step is done in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

/* softplus: the stable closed form of log(1 + exp(x)) ([S] MetalSelectiveScan; [K] step 2). */
double oracle_softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* silu(z) = z * sigmoid(z) ([K] step 6: out *= z * sigmoid(z)). */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Sequential forward recurrence for a list of (batch, channel) rows.
 *   rows[r] = b * Dm + d  (NULL: every row, in that order)
 *   h0 [batch, Dm, N] (NULL: zeros) is the state before step 0: h_{-1}[n] = h0[b, d, n].
 * Outputs (any may be NULL):
 *   y_rows    [nrows, L]  y[b, t, d]
 *   mag_rows  [nrows, L]  |silu(z)| * (sum_n |C_n h_t[n]| + |D u_t|): the size of the
 *                          terms that make up y, used as the denominator of the
 *                          condition-aware relative error
 *   last_rows [nrows, N]  h_{L-1}[n]
 * Per row, for t = 0..L-1 ([M] "Selective scan の本質", [K] "1チャンク内の処理フロー"):
 *   Δ_t     = softplus(delta_raw[b,t,d] + bias[d])
 *   h_t[n]  = exp(Δ_t · A_n) · h_{t-1}[n] + Δ_t · B[b,t,n] · u[b,t,d],  A_n = -exp(A_log[d,n])
 *   ŷ_t     = Σ_n C[b,t,n] · h_t[n] + D[d] · u[b,t,d]
 *   y[b,t,d]= ŷ_t · silu(z[b,t,d])   (ŷ_t when z is NULL)
 * The pre-softplus time step comes from delta_raw, or (delta_raw NULL) from the low-rank
 * projection dt_low [batch, L, R] · W_dt[Dm, R]^T summed in fp64 (see oracle_ss_fwd_dtproj_rows).
 */
static int fwd_rows(const float* u, const float* delta_raw, const float* dt_low, const float* W_dt, int64_t R,
                    const float* delta_bias, const float* A_log, const float* B, const float* C,
                    const float* D, const float* z, const double* h0, const int64_t* rows, int64_t nrows,
                    double* y_rows, double* mag_rows, double* last_rows,
                    int64_t batch, int64_t L, int64_t Dm, int64_t N)
{
    if (batch < 0 || L < 0 || Dm < 0 || N < 1) return ORACLE_EINVAL;
    if (!u || !A_log || !B || !C) return ORACLE_EINVAL;
    if (!delta_raw && (!dt_low || !W_dt || R < 1)) return ORACLE_EINVAL;
    if (rows == NULL) nrows = batch * Dm;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t row = rows ? rows[r] : r;
        if (row < 0 || row >= batch * Dm) {
#pragma omp atomic write
            status = ORACLE_EINVAL;
            continue;
        }
        const int64_t b = row / Dm, d = row % Dm;
        double* h = (double*)calloc((size_t)N, sizeof(double));
        double* A = (double*)malloc((size_t)N * sizeof(double));
        if (!h || !A) {
            free(h);
            free(A);
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int64_t n = 0; n < N; ++n) A[n] = -exp((double)A_log[d * N + n]);
        if (h0)
            for (int64_t n = 0; n < N; ++n) h[n] = h0[row * N + n];
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        const double Dd = D ? (double)D[d] : 0.0;

        for (int64_t t = 0; t < L; ++t) {
            const int64_t io = (b * L + t) * Dm + d;   /* [b, t, d] */
            const int64_t ib = (b * L + t) * N;        /* [b, t, 0] */
            const double ut = (double)u[io];
            double draw = 0.0;
            if (delta_raw) {
                draw = (double)delta_raw[io];
            } else {
                for (int64_t k = 0; k < R; ++k) draw += (double)W_dt[d * R + k] * (double)dt_low[(b * L + t) * R + k];
            }
            const double delta = oracle_softplus(draw + bias);
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                h[n] = exp(delta * A[n]) * h[n] + delta * (double)B[ib + n] * ut;
                const double ch = (double)C[ib + n] * h[n];
                acc += ch;
                acc_abs += fabs(ch);
            }
            const double skip = Dd * ut;
            const double gate = z ? oracle_silu((double)z[io]) : 1.0;
            if (y_rows) y_rows[r * L + t] = (acc + skip) * gate;
            if (mag_rows) mag_rows[r * L + t] = fabs(gate) * (acc_abs + fabs(skip));
        }
        if (last_rows)
            for (int64_t n = 0; n < N; ++n) last_rows[r * N + n] = h[n];
        free(h);
        free(A);
    }
    return status;
}

int oracle_ss_fwd_rows(const float* u, const float* delta_raw, const float* delta_bias,
                       const float* A_log, const float* B, const float* C, const float* D,
                       const float* z, const double* h0, const int64_t* rows, int64_t nrows,
                       double* y_rows, double* mag_rows, double* last_rows,
                       int64_t batch, int64_t L, int64_t Dm, int64_t N)
{
    if (!delta_raw) return ORACLE_EINVAL;
    return fwd_rows(u, delta_raw, NULL, NULL, 0, delta_bias, A_log, B, C, D, z, h0, rows, nrows,
                    y_rows, mag_rows, last_rows, batch, L, Dm, N);
}

/*
 * The forward scan with the time step's low-rank projection folded in: delta_raw[b,t,d] =
 * Σ_k W_dt[d,k] · dt_low[b,t,k] (k < R), summed in fp64, replaces the delta_raw input.  The
 * projection is the one SpeechLens kernel-optimization.md folds into its scan kernel (the
 * "dtProj–scan fusion" experiment: the rank-R delta projection computed inside the kernel
 * instead of materialising the [B, L, D] time steps).  dt_low [batch, L, R], W_dt [Dm, R].
 */
int oracle_ss_fwd_dtproj_rows(const float* u, const float* dt_low, const float* W_dt, int64_t R,
                              const float* delta_bias, const float* A_log, const float* B, const float* C,
                              const float* D, const float* z, const double* h0, const int64_t* rows,
                              int64_t nrows, double* y_rows, double* mag_rows, double* last_rows,
                              int64_t batch, int64_t L, int64_t Dm, int64_t N)
{
    if (!dt_low || !W_dt || R < 1) return ORACLE_EINVAL;
    return fwd_rows(u, NULL, dt_low, W_dt, R, delta_bias, A_log, B, C, D, z, h0, rows, nrows,
                    y_rows, mag_rows, last_rows, batch, L, Dm, N);
}

/*
 * The same forward result reached the way the scan method reaches it, in fp64:
 * per (row, state) the sequence is cut into chunks of `chunk` steps; inside a chunk
 * the pairs (a_t, b_t) = (exp(Δ_t A_n), Δ_t B_t,n u_t) are combined left to right with
 * the associative operator (a2,b2)∘(a1,b1) = (a2 a1, a2 b1 + b2) ([M] "Selective scan
 * の本質"; [K] "なぜ「scan」か"), and each chunk's running pair is applied to the carry
 * from the previous chunk, the carry being the state at the chunk's end ([M]
 * "チャンク間 running prefix").  It exists to check the oracle against itself:
 * any chunk length must give the sequential result up to rounding.  h0 (NULL: zeros) is
 * the carry before the first chunk.
 * Output layout as oracle_ss_fwd_rows (all rows, natural order).
 */
int oracle_ss_fwd_chunked(const float* u, const float* delta_raw, const float* delta_bias,
                          const float* A_log, const float* B, const float* C, const float* D,
                          const float* z, const double* h0, double* y_rows, double* last_rows,
                          int64_t batch, int64_t L, int64_t Dm, int64_t N, int64_t chunk)
{
    if (batch < 0 || L < 0 || Dm < 0 || N < 1 || chunk < 1) return ORACLE_EINVAL;
    const int64_t nrows = batch * Dm;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t row = 0; row < nrows; ++row) {
        const int64_t b = row / Dm, d = row % Dm;
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        const double Dd = D ? (double)D[d] : 0.0;
        double* pre = (double*)calloc((size_t)(L > 0 ? L : 1), sizeof(double));
        if (!pre) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int64_t n = 0; n < N; ++n) {
            const double An = -exp((double)A_log[d * N + n]);
            double carry = h0 ? h0[row * N + n] : 0.0;  /* state before the chunk */
            for (int64_t t0 = 0; t0 < L; t0 += chunk) {
                const int64_t t1 = (t0 + chunk < L) ? t0 + chunk : L;
                double run_a = 1.0, run_b = 0.0;      /* identity pair */
                for (int64_t t = t0; t < t1; ++t) {
                    const int64_t io = (b * L + t) * Dm + d;
                    const double delta = oracle_softplus((double)delta_raw[io] + bias);
                    const double a = exp(delta * An);
                    const double bb = delta * (double)B[(b * L + t) * N + n] * (double)u[io];
                    /* (a, bb) ∘ (run_a, run_b) */
                    run_b = a * run_b + bb;
                    run_a = a * run_a;
                    /* (run_a, run_b) ∘ (1, carry): the state at t */
                    const double h = run_a * carry + run_b;
                    pre[t] += (double)C[(b * L + t) * N + n] * h;
                }
                carry = run_a * carry + run_b;
            }
            if (last_rows) last_rows[row * N + n] = carry;
        }
        for (int64_t t = 0; t < L; ++t) {
            const int64_t io = (b * L + t) * Dm + d;
            const double gate = z ? oracle_silu((double)z[io]) : 1.0;
            if (y_rows) y_rows[row * L + t] = (pre[t] + Dd * (double)u[io]) * gate;
        }
        free(pre);
    }
    return status;
}

/*
 * Single-token decode update ([M] "O(L) インクリメンタルデコード"):
 *   Δ        = softplus(delta_raw[b,d] + bias[d])
 *   h[b,d,n] ← exp(Δ · A_n) · h[b,d,n] + Δ · x[b,d] · B[b,n]
 *   y[b,d]   = (Σ_n C[b,n] · h[b,d,n] + D[d] · x[b,d]) · silu(z[b,d])
 * state [batch, Dm, N] is read and overwritten in place (double).
 * x, delta_raw, z : [batch, Dm];  B, C : [batch, N].
 */
int oracle_ss_step(double* state, const float* x, const float* delta_raw,
                   const float* delta_bias, const float* A_log, const float* B,
                   const float* C, const float* D, const float* z,
                   double* y, double* mag, int64_t batch, int64_t Dm, int64_t N)
{
    if (batch < 0 || Dm < 0 || N < 1) return ORACLE_EINVAL;
    if (!state || !x || !delta_raw || !A_log || !B || !C) return ORACLE_EINVAL;

#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < batch * Dm; ++row) {
        const int64_t b = row / Dm, d = row % Dm;
        const double xt = (double)x[row];
        const double delta =
            oracle_softplus((double)delta_raw[row] + (delta_bias ? (double)delta_bias[d] : 0.0));
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double An = -exp((double)A_log[d * N + n]);
            double* h = &state[row * N + n];
            *h = exp(delta * An) * (*h) + delta * xt * (double)B[b * N + n];
            const double ch = (double)C[b * N + n] * (*h);
            acc += ch;
            acc_abs += fabs(ch);
        }
        const double skip = (D ? (double)D[d] : 0.0) * xt;
        const double gate = z ? oracle_silu((double)z[row]) : 1.0;
        if (y) y[row] = (acc + skip) * gate;
        if (mag) mag[row] = fabs(gate) * (acc_abs + fabs(skip));
    }
    return ORACLE_OK;
}

/*
 * Gradients of the forward scan (oracle_ss_fwd_rows with h0) for an upstream gradient dy of y
 * and dlast of last_state.  The pages implement no backward pass; this is the derivative of
 * the forward definition, written as the reverse (adjoint) recurrence of the same scan:
 *   g_t = silu(z_t) (1 without z),  yhat_t = sum_n C_t,n h_t,n + D u_t,  dyh_t = dy_t g_t
 *   dz_t = dy_t yhat_t silu'(z_t),  silu'(z) = s (1 + z (1 - s)),  s = sigmoid(z)
 *   lam_t,n = C_t,n dyh_t + a_{t+1},n lam_{t+1},n   (t = L-1 .. 0; dlast_n joins at t = L-1)
 *   dC_t,n += dyh_t h_t,n          dB_t,n += lam_t,n Delta_t u_t      (summed over channels)
 *   du_t = D dyh_t + sum_n lam_t,n Delta_t B_t,n
 *   dDelta_t = sum_n lam_t,n (A_n a_t,n h_{t-1},n + B_t,n u_t),  ddelta_raw_t = dDelta_t sigmoid(r_t)
 *   dA_n += sum_t lam_t,n Delta_t a_t,n h_{t-1},n,  dA_log = dA A,   dD += sum_t dyh_t u_t
 *   ddelta_bias += sum_t ddelta_raw_t,   dh0_n = a_0,n lam_0,n
 * with r_t = delta_raw + bias, Delta = softplus(r), A_n = -exp(A_log), a_t,n = exp(Delta_t A_n).
 * Inputs as oracle_ss_fwd_rows (h0 double, NULL = zeros); dy [batch, L, Dm] float; dlast
 * [batch, Dm, N] double or NULL.  Outputs (double, all written): du, ddelta_raw, dz
 * [batch, L, Dm]; dB, dC [batch, L, N]; dA_log [Dm, N]; dD, ddelta_bias [Dm]; dh0 [batch, Dm, N].
 * Parallel over batch rows (each owns its dB, dC); per-channel sums are combined after.
 */
int oracle_ss_bwd(const float* u, const float* delta_raw, const float* delta_bias,
                  const float* A_log, const float* B, const float* C, const float* D,
                  const float* z, const double* h0, const float* dy, const double* dlast,
                  double* du, double* ddelta_raw, double* dz, double* dB, double* dC,
                  double* dA_log, double* dD, double* ddelta_bias, double* dh0,
                  int64_t batch, int64_t L, int64_t Dm, int64_t N)
{
    if (batch < 0 || L < 0 || Dm < 0 || N < 1) return ORACLE_EINVAL;
    if (!u || !delta_raw || !A_log || !B || !C || !dy) return ORACLE_EINVAL;
    if (!du || !ddelta_raw || !dz || !dB || !dC || !dA_log || !dD || !ddelta_bias || !dh0) return ORACLE_EINVAL;
    /* per-batch-row partial sums of the per-channel gradients */
    double* pA = (double*)calloc((size_t)(batch > 0 ? batch : 1) * Dm * N, sizeof(double));
    double* pD = (double*)calloc((size_t)(batch > 0 ? batch : 1) * Dm, sizeof(double));
    double* pb = (double*)calloc((size_t)(batch > 0 ? batch : 1) * Dm, sizeof(double));
    if (!pA || !pD || !pb) {
        free(pA); free(pD); free(pb);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < batch * L * N; ++i) dB[i] = dC[i] = 0.0;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < batch; ++b) {
        double* hs = (double*)malloc((size_t)(L + 1) * N * sizeof(double));   /* h_{t-1} for t = 0..L */
        double* A = (double*)malloc((size_t)N * sizeof(double));
        double* lam = (double*)malloc((size_t)N * sizeof(double));
        if (!hs || !A || !lam) {
            free(hs); free(A); free(lam);
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int64_t d = 0; d < Dm; ++d) {
            const int64_t row = b * Dm + d;
            for (int64_t n = 0; n < N; ++n) A[n] = -exp((double)A_log[d * N + n]);
            const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
            const double Dd = D ? (double)D[d] : 0.0;
            /* forward: keep every state (hs row t+1 holds h_t, row 0 holds h_{-1}) */
            for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[row * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t io = (b * L + t) * Dm + d, ib = (b * L + t) * N;
                const double delta = oracle_softplus((double)delta_raw[io] + bias);
                for (int64_t n = 0; n < N; ++n)
                    hs[(t + 1) * N + n] = exp(delta * A[n]) * hs[t * N + n] + delta * (double)B[ib + n] * (double)u[io];
            }
            /* reverse */
            for (int64_t n = 0; n < N; ++n) lam[n] = dlast ? dlast[row * N + n] : 0.0;   /* a_{t+1} lam_{t+1} */
            for (int64_t t = L - 1; t >= 0; --t) {
                const int64_t io = (b * L + t) * Dm + d, ib = (b * L + t) * N;
                const double ut = (double)u[io];
                const double r = (double)delta_raw[io] + bias;
                const double delta = oracle_softplus(r);
                const double sig_r = 1.0 / (1.0 + exp(-r));
                double yhat = Dd * ut;
                for (int64_t n = 0; n < N; ++n) yhat += (double)C[ib + n] * hs[(t + 1) * N + n];
                double g = 1.0, dg = 0.0;
                if (z) {
                    const double zt = (double)z[io], s = 1.0 / (1.0 + exp(-zt));
                    g = zt * s;
                    dg = s * (1.0 + zt * (1.0 - s));
                }
                const double dyh = (double)dy[io] * g;
                dz[io] = z ? (double)dy[io] * yhat * dg : 0.0;
                double dut = Dd * dyh, ddel = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double l = (double)C[ib + n] * dyh + lam[n];
                    const double a = exp(delta * A[n]);
                    const double hp = hs[t * N + n];
                    dC[ib + n] += dyh * hs[(t + 1) * N + n];
                    dB[ib + n] += l * delta * ut;
                    dut += l * delta * (double)B[ib + n];
                    ddel += l * (A[n] * a * hp + (double)B[ib + n] * ut);
                    pA[row * N + n] += l * delta * a * hp;
                    lam[n] = a * l;
                }
                du[io] = dut;
                ddelta_raw[io] = ddel * sig_r;
                pD[row] += dyh * ut;
                pb[row] += ddel * sig_r;
            }
            for (int64_t n = 0; n < N; ++n) dh0[row * N + n] = lam[n];
        }
        free(hs); free(A); free(lam);
    }
    for (int64_t d = 0; d < Dm; ++d) {
        double sD = 0.0, sb = 0.0;
        for (int64_t b = 0; b < batch; ++b) {
            sD += pD[b * Dm + d];
            sb += pb[b * Dm + d];
        }
        dD[d] = sD;
        ddelta_bias[d] = sb;
        for (int64_t n = 0; n < N; ++n) {
            double sA = 0.0;
            for (int64_t b = 0; b < batch; ++b) sA += pA[(b * Dm + d) * N + n];
            dA_log[d * N + n] = sA * (-exp((double)A_log[d * N + n]));
        }
    }
    free(pA); free(pD); free(pb);
    return status;
}

/*
 * Causal depthwise convolution over the sequence, the stage before the scan in a Mamba block
 * ([M] "MambaBlock = in_proj -> conv1d -> SiLU -> ..."; [S] MetalCausalConv1d: depthwise,
 * kernel 4, three zero samples on the causal left edge, output length L), with the sliding
 * window that [M] "O(L) インクリメンタルデコード" carries across calls:
 *   pre[b,t,d] = bias[d] + sum_{k=0}^{K-1} w[d,k] * e[t + k],   e = window ++ x[b,:,d]
 *   out[b,t,d] = silu(pre) when act != 0, else pre
 * The window win_in[b,d,0..K-2] holds the K-1 samples before t = 0, oldest first (NULL: zeros,
 * i.e. the zero left padding).  win_out[b,d,:] receives the last K-1 samples of e, the window
 * a following call continues from.  Layouts: x [batch, L, Dm]; w [Dm, K]; bias [Dm] or NULL;
 * windows [batch, Dm, K-1]; out [batch, L, Dm].  Arithmetic in double.
 */
int oracle_conv1d(const float* x, const float* w, const float* bias, const double* win_in,
                  double* out, double* win_out, int64_t batch, int64_t L, int64_t Dm, int64_t K, int act)
{
    if (batch < 0 || L < 0 || Dm < 0 || K < 1) return ORACLE_EINVAL;
    if ((L > 0 && (!x || !out)) || !w) return ORACLE_EINVAL;
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t row = 0; row < batch * Dm; ++row) {
        const int64_t b = row / Dm, d = row % Dm;
        double* e = (double*)malloc((size_t)(L + K - 1) * sizeof(double));
        if (!e) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int64_t k = 0; k < K - 1; ++k) e[k] = win_in ? win_in[row * (K - 1) + k] : 0.0;
        for (int64_t t = 0; t < L; ++t) e[K - 1 + t] = (double)x[(b * L + t) * Dm + d];
        const double bd = bias ? (double)bias[d] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double acc = bd;
            for (int64_t k = 0; k < K; ++k) acc += (double)w[d * K + k] * e[t + k];
            out[(b * L + t) * Dm + d] = act ? oracle_silu(acc) : acc;
        }
        if (win_out)
            for (int64_t k = 0; k < K - 1; ++k) win_out[row * (K - 1) + k] = e[L + k];
        free(e);
    }
    return status;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
