/* Selective-scan oracle (fp64, sequential). TEST INFRASTRUCTURE ONLY: see mamba_oracle.c. */
#ifndef MAMBA_ORACLE_H
#define MAMBA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Forward over rows [row_begin, row_end), row = b * d_inner + d. Writes out (and y if non-null)
   at those rows only. Returns 0, 1 on bad arguments, 2 on allocation failure. */
int mamba_oracle_fwd_rows(const double* delta, const double* u, const double* B,
                          const double* C, const double* gate, const double* A_log,
                          const double* D, int64_t batch, int64_t T, int64_t d_inner,
                          int64_t d_state, int64_t row_begin, int64_t row_end, double* out,
                          double* y);

/* Forward + backward over rows [row_begin, row_end). Writes d_delta, d_u, d_gate at those
   rows; ADDS the rows' contributions into d_B_acc, d_C_acc [batch, T, d_state],
   d_A_log_acc [d_inner, d_state] and d_D_acc [d_inner]. */
int mamba_oracle_bwd_rows(const double* delta, const double* u, const double* B,
                          const double* C, const double* gate, const double* A_log,
                          const double* D, const double* dy, int64_t batch, int64_t T,
                          int64_t d_inner, int64_t d_state, int64_t row_begin, int64_t row_end,
                          double* d_delta, double* d_u, double* d_gate, double* d_B_acc,
                          double* d_C_acc, double* d_A_log_acc, double* d_D_acc);

/* Softplus of the raw delta, element-wise over n values: delta = raw for raw > 20, else
   log(1 + exp(raw)) (the threshold of mamba-rs src/mamba_ssm/cpu/backward.rs, "Softplus
   backward"; the forward is the function whose derivative that step takes). */
void mamba_oracle_softplus(const double* raw, double* delta, int64_t n);

/* Its backward: d_raw = d_delta for raw > 20, else d_delta * sigmoid(raw). */
void mamba_oracle_softplus_bwd(const double* raw, const double* d_delta, double* d_raw,
                               int64_t n);

/* Causal depthwise conv1d + SiLU, the step before the scan (mamba-rs
   src/mamba_ssm/cpu/backward.rs, Phase B6 is its backward). Forward, per (b, d):
     pre[t] = bias[d] + sum_{j<K} w[d, j] * x[t - (K-1) + j]     (x = 0 before t = 0)
     u[t]   = pre[t] * sigmoid(pre[t])
   x, u, pre: [batch, T, d_inner]; w: [d_inner, K]; bias: [d_inner]. pre may be NULL. */
int mamba_oracle_conv_fwd(const double* x, const double* w, const double* bias, int64_t batch,
                          int64_t T, int64_t d_inner, int64_t K, double* u, double* pre);

/* Backward, following Phase B6: d_pre = d_u * s * (1 + pre * (1 - s)); then, in reverse time,
   the current tap d_x[t] = d_pre[t] * w[d, K-1] plus the shift-register carry of later steps,
   and d_w[d, j] += d_pre[t] * x[t - (K-1) + j], d_bias[d] += d_pre[t]. d_x is written; d_w and
   d_bias are OVERWRITTEN with the sums over (b, t). */
int mamba_oracle_conv_bwd(const double* x, const double* w, const double* bias,
                          const double* d_u, int64_t batch, int64_t T, int64_t d_inner,
                          int64_t K, double* d_x, double* d_w, double* d_bias);

#ifdef __cplusplus
}
#endif
#endif
