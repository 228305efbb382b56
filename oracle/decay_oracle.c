/*
 * decay_oracle.c -- plain fp64 CPU oracle for the leaky (tau-decay) recurrent cell of the
 * pages' own model: forward recurrence, reverse-time backpropagation through time and the
 * gradients of W, b, tau, the inputs and the initial state.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file; only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes.  Page "K-loop Parallelization -- Block-per-Batch Kernel Refactor" names the
 * backward kernel's gradient scratch grad_w_in [B,128,128], grad_w_rec [B,128,128],
 * grad_b [B,128] and grad_tau [B,128] (section "Per-Kernel Breakdown") and a per-block vector
 * sdecay[n_hid] (section "Large shared-mem note"); it prints no equations.  The reading taken
 * is a leaky recurrence with one pre-activation per hidden unit and a decay per unit:
 *
 *     z_t  = [x_t ; h_{t-1}]              (n_in = n_x + C entries, h_{-1} = h0)
 *     a_t  = W z_t + b                    (W = [W_in | W_rec] is [C, n_in])
 *     e_t  = tanh(a_t)
 *     d_t  = exp(-ts[t,b] / tau)          (per hidden unit; tau > 0)
 *     h_t  = d_t * h_{t-1} + (1 - d_t) * e_t
 *
 * The backward pass is the vector-Jacobian product of L = sum_{t,b,i} dH[t,b,i] * H[t,b,i],
 * written out from the chain rule.  With G_t = dL/dh_t (dH[t] plus what flows back from t+1):
 *
 *     da_t      = G_t * (1 - d_t) * (1 - e_t^2)
 *     dz_t      = W^T da_t      ->  dx[t] = dz_t[0:n_x]
 *     G_{t-1}   = dH[t-1] + G_t * d_t + dz_t[n_x:]        (dh0 = G_t * d_t + dz_t[n_x:] at t=0)
 *     dtau     += G_t * (h_{t-1} - e_t) * d_t * ts[t,b] / tau^2    (d(d_t)/dtau = d_t ts / tau^2)
 *     dW       += da_t z_t^T,   db += da_t
 *
 * Layouts (row-major, last index fastest), all fp64:
 *   x [K][B][n_x], h0 [B][C], W [C][n_in], bias [C], tau [C], ts [K][B], dH [K][B][C],
 *   H [K][B][C], E [K][B][C] (tanh of the pre-activation), da [K][B][C], dW [C][n_in],
 *   db [C], dtau [C], dx [K][B][n_x], dh0 [B][C].
 *
 * Return value: 0 on success, -1 on a non-positive size or tau, -2 on an allocation failure.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* z_t for row b: [x_t ; h_{t-1}] with h_{-1} = h0. */
static void decay_gather_z(int B, int C, int n_x, int t, int b, const double* x, const double* h0,
                           const double* H, double* z) {
  const double* xr = x + ((size_t)t * B + b) * n_x;
  const double* hp = (t == 0) ? h0 + (size_t)b * C : H + ((size_t)(t - 1) * B + b) * C;
  memcpy(z, xr, sizeof(double) * n_x);
  memcpy(z + n_x, hp, sizeof(double) * C);
}

static int decay_check(int B, int K, int C, int n_x, const double* tau) {
  if (B <= 0 || K <= 0 || C <= 0 || n_x <= 0) return -1;
  for (int i = 0; i < C; ++i)
    if (!(tau[i] > 0.0)) return -1;
  return 0;
}

int cfc_decay_oracle_forward(int B, int K, int C, int n_x, const double* x, const double* h0,
                             const double* W, const double* bias, const double* tau,
                             const double* ts, double* H, double* E) {
  if (decay_check(B, K, C, n_x, tau) != 0) return -1;
  const int n_in = n_x + C;
  double* z = (double*)malloc(sizeof(double) * n_in);
  if (!z) return -2;
  for (int t = 0; t < K; ++t) {
    for (int b = 0; b < B; ++b) {
      decay_gather_z(B, C, n_x, t, b, x, h0, H, z);
      const double* hp = z + n_x;
      const double dt = ts[(size_t)t * B + b];
      double* ho = H + ((size_t)t * B + b) * C;
      double* eo = E + ((size_t)t * B + b) * C;
      for (int i = 0; i < C; ++i) {
        double a = bias[i];
        const double* wr = W + (size_t)i * n_in;
        for (int k = 0; k < n_in; ++k) a += wr[k] * z[k];
        const double e = tanh(a);
        const double d = exp(-dt / tau[i]);
        eo[i] = e;
        ho[i] = d * hp[i] + (1.0 - d) * e;
      }
    }
  }
  free(z);
  return 0;
}

int cfc_decay_oracle_backward(int B, int K, int C, int n_x, const double* x, const double* h0,
                              const double* W, const double* tau, const double* ts,
                              const double* H, const double* E, const double* dH, double* da,
                              double* dW, double* db, double* dtau, double* dx, double* dh0) {
  if (decay_check(B, K, C, n_x, tau) != 0) return -1;
  const int n_in = n_x + C;
  double* z = (double*)malloc(sizeof(double) * n_in);
  double* G = (double*)malloc(sizeof(double) * C);
  double* dz = (double*)malloc(sizeof(double) * n_in);
  if (!z || !G || !dz) {
    free(z);
    free(G);
    free(dz);
    return -2;
  }
  memset(dW, 0, sizeof(double) * C * n_in);
  memset(db, 0, sizeof(double) * C);
  memset(dtau, 0, sizeof(double) * C);
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < C; ++i) G[i] = 0.0;
    for (int t = K - 1; t >= 0; --t) {
      decay_gather_z(B, C, n_x, t, b, x, h0, H, z);
      const double* hp = z + n_x;
      const double dt = ts[(size_t)t * B + b];
      const double* dHt = dH + ((size_t)t * B + b) * C;
      const double* et = E + ((size_t)t * B + b) * C;
      double* dat = da + ((size_t)t * B + b) * C;
      for (int i = 0; i < C; ++i) G[i] += dHt[i];  /* G_t = dH[t] + flow from t+1 */
      for (int i = 0; i < C; ++i) {
        const double d = exp(-dt / tau[i]);
        dat[i] = G[i] * (1.0 - d) * (1.0 - et[i] * et[i]);
        dtau[i] += G[i] * (hp[i] - et[i]) * d * dt / (tau[i] * tau[i]);
      }
      for (int k = 0; k < n_in; ++k) dz[k] = 0.0;
      for (int i = 0; i < C; ++i) {
        const double* wr = W + (size_t)i * n_in;
        for (int k = 0; k < n_in; ++k) dz[k] += wr[k] * dat[i];
      }
      for (int i = 0; i < C; ++i) {
        double* dwr = dW + (size_t)i * n_in;
        for (int k = 0; k < n_in; ++k) dwr[k] += dat[i] * z[k];
        db[i] += dat[i];
      }
      double* dxt = dx + ((size_t)t * B + b) * n_x;
      for (int k = 0; k < n_x; ++k) dxt[k] = dz[k];
      for (int i = 0; i < C; ++i) G[i] = G[i] * exp(-dt / tau[i]) + dz[n_x + i];
    }
    for (int i = 0; i < C; ++i) dh0[(size_t)b * C + i] = G[i];
  }
  free(z);
  free(G);
  free(dz);
  return 0;
}

double cfc_decay_oracle_loss(int B, int K, int C, const double* H, const double* dH) {
  double s = 0.0;
  const size_t n = (size_t)K * B * C;
  for (size_t i = 0; i < n; ++i) s += dH[i] * H[i];
  return s;
}
