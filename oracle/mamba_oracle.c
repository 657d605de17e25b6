/*
 * Selective-scan oracle: fp64, single-threaded, sequential in t.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU-baseline leg
 * load this file; the CUDA library never does, and it shares no code with it.
 *
 * What it computes, per independent row (b, d), with A[d,n] = -exp(A_log[d,n]):
 *
 *   forward   h_{-1}[n] = 0
 *             da_t[n]   = exp(delta_t * A[n])
 *             h_t[n]    = da_t[n] * h_{t-1}[n] + delta_t * u_t * B_t[n]
 *             y_t       = sum_n C_t[n] * h_t[n] + D * u_t
 *             out_t     = y_t * gate_t * sigmoid(gate_t)               (y * SiLU(gate))
 *
 *   backward  the gating backward (mamba-rs src/mamba_ssm/cpu/backward.rs, Phase B2) and the
 *             reverse-time SSM BPTT (same file, Phase B3), taken step by step in that order:
 *             d_y = dy * SiLU(g);  d_gate = dy * y * s * (1 + g * (1 - s)),  s = sigmoid(g);
 *             then for t = T-1 .. 0, with d_h starting at zero:
 *               d_D += d_y * u;  d_u = d_y * D
 *               for each n:  d_h[n] += d_y * C[n]
 *                            d_delta += d_h[n] * (A[n] * da[n] * h_prev[n] + u * B[n])
 *                            d_u     += d_h[n] * delta * B[n]
 *                            d_B[n]  += d_h[n] * delta * u
 *                            d_C[n]  += d_y * h[n]
 *                            d_A_log[n] += d_h[n] * da[n] * delta * A[n] * h_prev[n]
 *                            d_h[n]  = da[n] * d_h[n]
 *
 * The forward recurrence itself is not printed on the page; it is the one whose partial
 * derivatives the Phase B3 updates are (dh/dB = delta*u, dh/du = delta*B, dh/ddelta contains
 * u*B and A*da*h_prev), with a zero initial state.
 *
 * Layouts (row-major, contiguous): delta, u, gate, dy, out, y, d_delta, d_u, d_gate are
 * [batch, T, d_inner]; B, C, d_B, d_C are [batch, T, d_state]; A_log, d_A_log are
 * [d_inner, d_state]; D, d_D are [d_inner].
 *
 * Rows are row = b * d_inner + d. The *_rows entry points process rows [row_begin, row_end):
 * they write the per-row outputs of those rows and ADD the rows' contributions into the
 * d_B, d_C, d_A_log, d_D accumulators, so that a caller may split the rows across threads,
 * each with its own accumulators, and sum the accumulators afterwards.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "mamba_oracle.h"

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

int mamba_oracle_fwd_rows(const double* delta, const double* u, const double* Bm,
                          const double* Cm, const double* gate, const double* A_log,
                          const double* Dp, int64_t batch, int64_t T, int64_t Di, int64_t N,
                          int64_t row_begin, int64_t row_end, double* out, double* y) {
  if (batch <= 0 || T <= 0 || Di <= 0 || N <= 0) return 1;
  if (row_begin < 0 || row_end > batch * Di || row_begin > row_end) return 1;
  double* h = (double*)calloc((size_t)N, sizeof(double));
  double* A = (double*)malloc((size_t)N * sizeof(double));
  if (!h || !A) { free(h); free(A); return 2; }
  for (int64_t row = row_begin; row < row_end; ++row) {
    const int64_t b = row / Di, d = row % Di;
    for (int64_t n = 0; n < N; ++n) { A[n] = -exp(A_log[d * N + n]); h[n] = 0.0; }
    for (int64_t t = 0; t < T; ++t) {
      const int64_t bt = b * T + t;
      const int64_t i = bt * Di + d;
      double yv = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double da = exp(delta[i] * A[n]);
        h[n] = da * h[n] + delta[i] * u[i] * Bm[bt * N + n];
        yv += Cm[bt * N + n] * h[n];
      }
      yv += Dp[d] * u[i];
      if (y) y[i] = yv;
      const double g = gate[i];
      out[i] = yv * g * sigmoid(g);
    }
  }
  free(h);
  free(A);
  return 0;
}

int mamba_oracle_bwd_rows(const double* delta, const double* u, const double* Bm,
                          const double* Cm, const double* gate, const double* A_log,
                          const double* Dp, const double* dy, int64_t batch, int64_t T,
                          int64_t Di, int64_t N, int64_t row_begin, int64_t row_end,
                          double* d_delta, double* d_u, double* d_gate, double* d_B_acc,
                          double* d_C_acc, double* d_A_log_acc, double* d_D_acc) {
  if (batch <= 0 || T <= 0 || Di <= 0 || N <= 0) return 1;
  if (row_begin < 0 || row_end > batch * Di || row_begin > row_end) return 1;
  /* The row's whole forward trajectory, as the page's stored activations hold it:
     h for every t (h_curr; h_prev is the previous row of it), da for every t, and y. */
  double* H = (double*)malloc((size_t)(T * N) * sizeof(double));
  double* DA = (double*)malloc((size_t)(T * N) * sizeof(double));
  double* Y = (double*)malloc((size_t)T * sizeof(double));
  double* A = (double*)malloc((size_t)N * sizeof(double));
  double* dh = (double*)malloc((size_t)N * sizeof(double));
  if (!H || !DA || !Y || !A || !dh) { free(H); free(DA); free(Y); free(A); free(dh); return 2; }

  for (int64_t row = row_begin; row < row_end; ++row) {
    const int64_t b = row / Di, d = row % Di;
    for (int64_t n = 0; n < N; ++n) A[n] = -exp(A_log[d * N + n]);

    /* forward, keeping the trajectory */
    for (int64_t t = 0; t < T; ++t) {
      const int64_t bt = b * T + t;
      const int64_t i = bt * Di + d;
      double yv = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double hp = (t > 0) ? H[(t - 1) * N + n] : 0.0;
        const double da = exp(delta[i] * A[n]);
        const double hc = da * hp + delta[i] * u[i] * Bm[bt * N + n];
        DA[t * N + n] = da;
        H[t * N + n] = hc;
        yv += Cm[bt * N + n] * hc;
      }
      Y[t] = yv + Dp[d] * u[i];
    }

    /* Phase B2 gating backward and Phase B3 reverse SSM BPTT, per the page's order */
    for (int64_t n = 0; n < N; ++n) dh[n] = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      const int64_t bt = b * T + t;
      const int64_t i = bt * Di + d;
      const double g = gate[i];
      const double s = sigmoid(g);
      const double d_gated = dy[i];
      const double dyv = d_gated * (g * s);                 /* d_y = d_gated * SiLU(gate)   */
      d_gate[i] = d_gated * Y[t] * (s * (1.0 + g * (1.0 - s)));

      const double dl = delta[i], uu = u[i];
      d_D_acc[d] += dyv * uu;
      double du = dyv * Dp[d];
      double ddl = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double bn = Bm[bt * N + n];
        const double cn = Cm[bt * N + n];
        const double da = DA[t * N + n];
        const double hp = (t > 0) ? H[(t - 1) * N + n] : 0.0;
        const double hc = H[t * N + n];
        dh[n] += dyv * cn;
        const double g_h = dh[n];
        ddl += g_h * (A[n] * da * hp + uu * bn);
        du += g_h * dl * bn;
        d_B_acc[bt * N + n] += g_h * dl * uu;
        d_C_acc[bt * N + n] += dyv * hc;
        d_A_log_acc[d * N + n] += g_h * da * dl * A[n] * hp;
        dh[n] = da * g_h;
      }
      d_delta[i] = ddl;
      d_u[i] = du;
    }
  }
  free(H);
  free(DA);
  free(Y);
  free(A);
  free(dh);
  return 0;
}

/* Softplus with the threshold 20 of mamba-rs src/mamba_ssm/cpu/backward.rs ("Softplus
   backward"): the identity above it, log(1 + e^x) below. */
void mamba_oracle_softplus(const double* raw, double* delta, int64_t n) {
  for (int64_t i = 0; i < n; ++i) delta[i] = raw[i] > 20.0 ? raw[i] : log1p(exp(raw[i]));
}

/* The derivative of softplus is the logistic sigmoid; above the threshold it is 1 (same
   passage). */
void mamba_oracle_softplus_bwd(const double* raw, const double* d_delta, double* d_raw,
                               int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    d_raw[i] = raw[i] > 20.0 ? d_delta[i] : d_delta[i] * (1.0 / (1.0 + exp(-raw[i])));
}

/* ---- causal depthwise conv1d + SiLU (the step before the scan) ---------------------------- */
/* Forward: the shift register of the last K inputs of channel d, dotted with w[d, :]. */
int mamba_oracle_conv_fwd(const double* x, const double* w, const double* bias, int64_t batch,
                          int64_t T, int64_t d_inner, int64_t K, double* u, double* pre) {
  if (batch < 1 || T < 1 || d_inner < 1 || K < 1 || !x || !w || !bias || !u) return 1;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t d = 0; d < d_inner; ++d)
      for (int64_t t = 0; t < T; ++t) {
        double acc = bias[d];
        for (int64_t j = 0; j < K; ++j) {
          const int64_t ts = t - (K - 1) + j;
          if (ts >= 0) acc += w[d * K + j] * x[(b * T + ts) * d_inner + d];
        }
        const double s = 1.0 / (1.0 + exp(-acc));
        const int64_t i = (b * T + t) * d_inner + d;
        u[i] = acc * s;
        if (pre) pre[i] = acc;
      }
  return 0;
}

/* Backward (Phase B6): SiLU backward for every t, then the reverse pass with the carry. The
   carry of channel d holds, for the next (earlier) step, sum_{m>=1} d_pre[t+m] * w[d, K-1-m];
   it shifts by one tap per step. */
int mamba_oracle_conv_bwd(const double* x, const double* w, const double* bias,
                          const double* d_u, int64_t batch, int64_t T, int64_t d_inner,
                          int64_t K, double* d_x, double* d_w, double* d_bias) {
  if (batch < 1 || T < 1 || d_inner < 1 || K < 1 || !x || !w || !bias || !d_u || !d_x || !d_w ||
      !d_bias)
    return 1;
  double* pre = (double*)malloc(sizeof(double) * (size_t)(batch * T * d_inner));
  double* u = (double*)malloc(sizeof(double) * (size_t)(batch * T * d_inner));
  double* carry = (double*)calloc((size_t)(K > 1 ? K - 1 : 1), sizeof(double));
  if (!pre || !u || !carry) {
    free(pre); free(u); free(carry);
    return 2;
  }
  mamba_oracle_conv_fwd(x, w, bias, batch, T, d_inner, K, u, pre);
  for (int64_t i = 0; i < d_inner * K; ++i) d_w[i] = 0.0;
  for (int64_t d = 0; d < d_inner; ++d) d_bias[d] = 0.0;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t d = 0; d < d_inner; ++d) {
      for (int64_t k = 0; k + 1 < K; ++k) carry[k] = 0.0;
      for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t i = (b * T + t) * d_inner + d;
        const double p = pre[i];
        const double s = 1.0 / (1.0 + exp(-p));
        const double dp = d_u[i] * s * (1.0 + p * (1.0 - s));
        /* this step's tap and the parameter gradients (the register holds x[t-K+1 .. t]) */
        double dx = dp * w[d * K + (K - 1)];
        for (int64_t j = 0; j < K; ++j) {
          const int64_t ts = t - (K - 1) + j;
          if (ts >= 0) d_w[d * K + j] += dp * x[(b * T + ts) * d_inner + d];
        }
        d_bias[d] += dp;
        /* carry from later steps, then shift it and add this step's taps for earlier steps */
        if (K > 1) {
          dx += carry[0];
          for (int64_t k = 0; k + 2 < K; ++k) carry[k] = carry[k + 1] + dp * w[d * K + (K - 2 - k)];
          carry[K - 2] = dp * w[d * K + 0];
        }
        d_x[i] = dx;
      }
    }
  free(pre);
  free(u);
  free(carry);
  return 0;
}
