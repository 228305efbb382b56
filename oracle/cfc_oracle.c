/*
 * cfc_oracle.c -- plain fp64 CPU oracle for the CfC K-loop: forward recurrence, reverse-time
 * backpropagation through time, weight/bias/input/initial-state gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file; only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes.  The K-loop parallelization spec (page "K-loop Parallelization --
 * Block-per-Batch Kernel Refactor", section "Problem") names the forward kernel
 * cfc_step_batched (one CfC step for the whole batch, called once per K step) and the backward
 * kernel cfc_step_backward_batched (one reverse step, called once per K step), but does not
 * print the cell's equations.  The cell used here is the four-gate closed-form continuous-time
 * cell:
 *
 *     z_t  = [u_t ; h_{t-1}]                       (n_in = n_x + C entries, h_{-1} = h0)
 *     P_g  = W_g z_t + b_g        for g in {ff1, ff2, ta, tb}   (each W_g is [C, n_in])
 *     ff1  = tanh(P_ff1),  ff2 = tanh(P_ff2)
 *     gate = sigmoid(P_ta * ts[t,b] + P_tb),  sigmoid(x) = 1 / (1 + exp(-x))
 *     h_t  = ff1 * (1 - gate) + gate * ff2
 *
 * The backward pass is the vector-Jacobian product of the scalar L = sum_{t,b,i} dH[t,b,i] *
 * H[t,b,i], written out by hand from the chain rule (no reordering beyond the definition):
 *
 *     dh      = dH[t] + delta_t          (delta_{K-1} = 0)
 *     dP_ff1  = dh * (1 - gate) * (1 - ff1^2)
 *     dP_ff2  = dh * gate * (1 - ff2^2)
 *     ds      = dh * (ff2 - ff1) * gate * (1 - gate)
 *     dP_ta   = ds * ts[t,b],   dP_tb = ds
 *     dz      = sum_g W_g^T dP_g     ->  du[t] = dz[0:n_x],  delta_{t-1} = dz[n_x:]
 *     dh0     = delta_{-1}
 *     dW_g    = sum_{t,b} dP_g[t,b] z_t[b]^T,   db_g = sum_{t,b} dP_g[t,b]
 *
 * The weight gradient is the dense sum over batch and time that the DQN plan (page "H100 Epoch
 * Optimization Phase 2", Task 2) describes as dW = dY^T X in place of per-sample atomic
 * accumulation; here it is a plain triple loop in fp64.
 *
 * Layouts (row-major, last index fastest), all fp64:
 *   u [K][B][n_x], h0 [B][C], W [4][C][n_in], bias [4][C], ts [K][B], dH [K][B][C],
 *   H [K][B][C], ff1/ff2/gate [K][B][C], d_pre [K][B][4][C], dW [4][C][n_in], db [4][C],
 *   du [K][B][n_x], dh0 [B][C].
 *
 * Return value: 0 on success, -1 on a non-positive size, -2 on an allocation failure.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* z_t[b] = [u[t][b] ; h_{t-1}[b]] with h_{-1} = h0. */
static void gather_z(int B, int C, int n_x, int t, int b, const double* u, const double* h0,
                     const double* H, double* z) {
    const double* hprev = (t == 0) ? &h0[(size_t)b * C] : &H[((size_t)(t - 1) * B + b) * C];
    for (int k = 0; k < n_x; ++k) z[k] = u[((size_t)t * B + b) * n_x + k];
    for (int j = 0; j < C; ++j) z[n_x + j] = hprev[j];
}

/* Forward recurrence over t = 0..K-1 for every batch row.  ff1/ff2/gate may be NULL. */
int cfc_oracle_forward(int B, int K, int C, int n_x, const double* u, const double* h0,
                       const double* W, const double* bias, const double* ts, double* H,
                       double* ff1_out, double* ff2_out, double* gate_out) {
    if (B <= 0 || K <= 0 || C <= 0 || n_x <= 0) return -1;
    const int n_in = n_x + C;
    double* z = (double*)malloc(sizeof(double) * (size_t)n_in);
    if (!z) return -2;
    for (int t = 0; t < K; ++t) {
        for (int b = 0; b < B; ++b) {
            gather_z(B, C, n_x, t, b, u, h0, H, z);
            for (int i = 0; i < C; ++i) {
                double P[4];
                for (int g = 0; g < 4; ++g) {
                    const double* w = &W[((size_t)g * C + i) * n_in];
                    double acc = bias[(size_t)g * C + i];
                    for (int k = 0; k < n_in; ++k) acc += w[k] * z[k];
                    P[g] = acc;
                }
                const double f1 = tanh(P[0]);
                const double f2 = tanh(P[1]);
                const double gt = sigmoid(P[2] * ts[(size_t)t * B + b] + P[3]);
                const size_t o = ((size_t)t * B + b) * C + i;
                H[o] = f1 * (1.0 - gt) + gt * f2;
                if (ff1_out) ff1_out[o] = f1;
                if (ff2_out) ff2_out[o] = f2;
                if (gate_out) gate_out[o] = gt;
            }
        }
    }
    free(z);
    return 0;
}

/* L = sum dH * H (the scalar whose gradient the backward pass returns). */
double cfc_oracle_loss(int B, int K, int C, const double* H, const double* dH) {
    double acc = 0.0;
    const size_t n = (size_t)K * B * C;
    for (size_t e = 0; e < n; ++e) acc += dH[e] * H[e];
    return acc;
}

/* Reverse-time BPTT, then the weight, bias and input gradients.  d_pre may be NULL. */
int cfc_oracle_backward(int B, int K, int C, int n_x, const double* u, const double* h0,
                        const double* W, const double* ts, const double* H, const double* ff1,
                        const double* ff2, const double* gate, const double* dH,
                        double* d_pre_out, double* dW, double* db, double* du, double* dh0) {
    if (B <= 0 || K <= 0 || C <= 0 || n_x <= 0) return -1;
    const int n_in = n_x + C;
    const size_t n_pre = (size_t)K * B * 4 * C;
    double* d_pre = d_pre_out ? d_pre_out : (double*)malloc(sizeof(double) * n_pre);
    double* delta = (double*)calloc((size_t)B * C, sizeof(double));
    double* dz = (double*)malloc(sizeof(double) * (size_t)n_in);
    double* z = (double*)malloc(sizeof(double) * (size_t)n_in);
    if (!d_pre || !delta || !dz || !z) {
        if (!d_pre_out) free(d_pre);
        free(delta); free(dz); free(z);
        return -2;
    }

    /* Reverse-time recurrence: d_pre[t] from dh = dH[t] + delta, then delta <- W_h^T d_pre[t]. */
    for (int t = K - 1; t >= 0; --t) {
        for (int b = 0; b < B; ++b) {
            const size_t row = (size_t)t * B + b;
            double* dp = &d_pre[row * 4 * C];
            const double tsv = ts[row];
            for (int i = 0; i < C; ++i) {
                const size_t o = row * C + i;
                const double dh = dH[o] + delta[(size_t)b * C + i];
                const double f1 = ff1[o], f2 = ff2[o], gt = gate[o];
                const double ds = dh * (f2 - f1) * gt * (1.0 - gt);
                dp[0 * C + i] = dh * (1.0 - gt) * (1.0 - f1 * f1);
                dp[1 * C + i] = dh * gt * (1.0 - f2 * f2);
                dp[2 * C + i] = ds * tsv;
                dp[3 * C + i] = ds;
            }
            for (int k = 0; k < n_in; ++k) {
                double acc = 0.0;
                for (int g = 0; g < 4; ++g)
                    for (int i = 0; i < C; ++i)
                        acc += W[((size_t)g * C + i) * n_in + k] * dp[g * C + i];
                dz[k] = acc;
            }
            for (int k = 0; k < n_x; ++k) du[row * n_x + k] = dz[k];
            for (int j = 0; j < C; ++j) delta[(size_t)b * C + j] = dz[n_x + j];
        }
    }
    memcpy(dh0, delta, sizeof(double) * (size_t)B * C);

    /* dW_g = sum_{t,b} dP_g z^T and db_g = sum_{t,b} dP_g, summed in (t, b) order. */
    memset(dW, 0, sizeof(double) * (size_t)4 * C * n_in);
    memset(db, 0, sizeof(double) * (size_t)4 * C);
    for (int t = 0; t < K; ++t) {
        for (int b = 0; b < B; ++b) {
            const size_t row = (size_t)t * B + b;
            gather_z(B, C, n_x, t, b, u, h0, H, z);
            const double* dp = &d_pre[row * 4 * C];
            for (int m = 0; m < 4 * C; ++m) {
                const double a = dp[m];
                double* dw = &dW[(size_t)m * n_in];
                for (int k = 0; k < n_in; ++k) dw[k] += a * z[k];
                db[m] += a;
            }
        }
    }

    if (!d_pre_out) free(d_pre);
    free(delta); free(dz); free(z);
    return 0;
}

/* Plain sum over axis 0 of a [n_batch][n_tail] array in batch-index order (fp64). */
int cfc_oracle_reduce_axis0(int n_batch, int n_tail, const double* per_batch, double* out) {
    if (n_batch <= 0 || n_tail <= 0) return -1;
    for (int n = 0; n < n_tail; ++n) out[n] = 0.0;
    for (int r = 0; r < n_batch; ++r)
        for (int n = 0; n < n_tail; ++n) out[n] += per_batch[(size_t)r * n_tail + n];
    return 0;
}
