/*
 * ssm_oracle.c -- the CPU oracle: plain sequential loops in double precision.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  No blocking, no
 * fusion, no reordering beyond what the definitions state.
 *
 * Sources (web pages the method is taken from):
 *  - ggmlR tests/testthat/test-ssm-rwkv.R: the ssm_conv definition (test "ggml_ssm_conv
 *    matches a depthwise convolution computed in R"), the ssm_scan operand shapes
 *    (helper make_scan) and the packed results of ssm_scan / ssm_conv_back / ssm_scan_back.
 *  - infotheory backends/mambazip/mamba1/model.rs: the per-token selective scan
 *    (forward_impl and selective_scan_state16), silu / softplus / silu_grad_from_sigmoid,
 *    the per-token adjoint (accumulate_token_step_gradients) and the TBPTT replay with
 *    per-chunk checkpoints (online_train_segment_tbptt).
 *  - kizzasi-model src/backprop_ssm.rs: the reverse adjoint scan and the initial-state
 *    gradient (ssm_backward), the affine-scan composition (associative_scan_backward) and
 *    segment checkpoints (GradientCheckpointedSSM).
 *  - lattice-inference src/attention/gdn_backward.rs: causal conv1d + SiLU forward
 *    (conv1d_silu_fwd) and its lag-scatter backward (step 5 of gdn_backward).
 */
#include "ssm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- pointwise functions (infotheory model.rs: silu, sigmoid, softplus,
 *      silu_grad_from_sigmoid) ------------------------------------------------ */
static double sigmoid_d(double v) { return 1.0 / (1.0 + exp(-v)); }
static double silu_d(double v) { return v * sigmoid_d(v); }
static double silu_grad_d(double v) {
  double s = sigmoid_d(v);
  return s * (1.0 + v * (1.0 - s));
}
/* softplus with the page's threshold: identity above 20 */
static double softplus_d(double v) { return v > 20.0 ? v : log1p(exp(v)); }
/* derivative of that piecewise function */
static double softplus_grad_d(double v) { return v > 20.0 ? 1.0 : sigmoid_d(v); }

/* ---- causal depthwise conv1d (+ optional bias and SiLU) -----------------------
 * ggmlR test-ssm-rwkv.R, "ggml_ssm_conv matches a depthwise convolution computed in R":
 * output position t of channel ch sums the d_conv taps sx[ch][t + j] * c[ch][j], so the
 * last tap multiplies the newest input (as in conv1d_silu_fwd of gdn_backward.rs).  The
 * bias and SiLU are the Mamba-1 additions of infotheory model.rs (depthwise_conv_step,
 * then silu). */
int oracle_conv_fwd(const double* sx, const double* c, const double* bias, double* out,
                    double* conv_state_out, int n_s, int d_inner, int n_t, int d_conv, int silu) {
  if (n_s <= 0 || d_inner <= 0 || n_t <= 0 || d_conv <= 0) return -1;
  const long W = (long)n_t + d_conv - 1;
  for (int b = 0; b < n_s; b++)
    for (int t = 0; t < n_t; t++)
      for (int d = 0; d < d_inner; d++) {
        const double* row = sx + ((long)b * d_inner + d) * W;
        double acc = 0.0;
        for (int k = 0; k < d_conv; k++) acc += row[t + k] * c[(long)d * d_conv + k];
        if (bias) acc += bias[d];
        out[((long)b * n_t + t) * d_inner + d] = silu ? silu_d(acc) : acc;
      }
  if (conv_state_out) /* the K-1 newest columns: the rolling state a next call starts from */
    for (int b = 0; b < n_s; b++)
      for (int d = 0; d < d_inner; d++)
        for (int k = 0; k < d_conv - 1; k++)
          conv_state_out[((long)b * d_inner + d) * (d_conv - 1) + k] =
              sx[((long)b * d_inner + d) * W + n_t + k];
  return 0;
}

/* Reverse mode of the above.  gdn_backward.rs step 5: recompute the pre-activation,
 * multiply by SiLU', then scatter d_sum * w[tap] back to the input column the tap read.
 * ggmlR packs the results as [d_sx | d_c] ("ggml_ssm_conv_back packs both input gradients"). */
int oracle_conv_bwd(const double* sx, const double* c, const double* bias, const double* dout,
                    double* d_sx, double* d_c, double* d_bias,
                    int n_s, int d_inner, int n_t, int d_conv, int silu) {
  if (n_s <= 0 || d_inner <= 0 || n_t <= 0 || d_conv <= 0) return -1;
  const long W = (long)n_t + d_conv - 1;
  memset(d_sx, 0, sizeof(double) * (size_t)n_s * d_inner * W);
  memset(d_c, 0, sizeof(double) * (size_t)d_inner * d_conv);
  if (d_bias) memset(d_bias, 0, sizeof(double) * (size_t)d_inner);
  for (int b = 0; b < n_s; b++)
    for (int t = 0; t < n_t; t++)
      for (int d = 0; d < d_inner; d++) {
        const double* row = sx + ((long)b * d_inner + d) * W;
        double pre = 0.0;
        for (int k = 0; k < d_conv; k++) pre += row[t + k] * c[(long)d * d_conv + k];
        if (bias) pre += bias[d];
        double g = dout[((long)b * n_t + t) * d_inner + d];
        if (silu) g *= silu_grad_d(pre);
        for (int k = 0; k < d_conv; k++) {
          d_sx[((long)b * d_inner + d) * W + t + k] += g * c[(long)d * d_conv + k];
          d_c[(long)d * d_conv + k] += g * row[t + k];
        }
        if (d_bias) d_bias[d] += g;
      }
  return 0;
}

/* ---- selective scan ------------------------------------------------------------ */

static int dims_ok(const oracle_scan_dims* m) {
  if (!m) return 0;
  if (m->n_seqs <= 0 || m->n_tok <= 0 || m->n_head <= 0 || m->head_dim <= 0 || m->d_state <= 0 ||
      m->n_group <= 0 || m->chunk <= 0)
    return 0;
  if (m->n_head % m->n_group != 0) return 0;
  return 1;
}

/* row of s0 / d_s0 that sequence b starts from ("one state row each", make_scan) */
static int state_row(const int* ids, int b) { return ids ? ids[b] : b; }

/* delta for (b, t, h): dt as given, or softplus(dt + dt_bias) (forward_impl: dt_pre -> softplus) */
static double delta_at(const oracle_scan_dims* m, const double* dt, const double* dt_bias, int b,
                       int t, int h, double* pre_out) {
  double v = dt[((long)b * m->n_tok + t) * m->n_head + h];
  if (m->dt_softplus) {
    if (dt_bias) v += dt_bias[h];
    if (pre_out) *pre_out = v;
    return softplus_d(v);
  }
  if (pre_out) *pre_out = v;
  return v;
}

static double a_coef(const oracle_scan_dims* m, const double* A, int h, int n) {
  return m->a_per_state ? A[(long)h * m->d_state + n] : A[h];
}

/* One forward step of the recurrence for channel (b, h, p) at token t, all N states
 * (selective_scan_state16 / forward_impl of infotheory model.rs):
 *   a = exp(delta * A),  h_t = a * h_{t-1} + (delta * x) * B_t,
 * returns y_pre = sum_n C_t[n] h_t[n] + D * x (the gate is applied by the caller). */
static double step_fwd(const oracle_scan_dims* m, int b, int t, int h, int p, const double* x,
                       const double* A, const double* B, const double* C, const double* D,
                       double delta, const double* h_prev, double* h_new) {
  const int H = m->n_head, P = m->head_dim, N = m->d_state, G = m->n_group, L = m->n_tok;
  const int g = h / (H / G);
  const double xv = x[(((long)b * L + t) * H + h) * P + p];
  const double* Bt = B + (((long)b * L + t) * G + g) * N;
  const double* Ct = C + (((long)b * L + t) * G + g) * N;
  double acc = 0.0;
  for (int n = 0; n < N; n++) {
    double a = exp(delta * a_coef(m, A, h, n));
    h_new[n] = a * h_prev[n] + (delta * xv) * Bt[n];
    acc += Ct[n] * h_new[n];
  }
  if (D) acc += D[h * P + p] * xv;
  return acc;
}

int oracle_scan_fwd(const oracle_scan_dims* m, const double* s0, const int* ids, const double* x,
                    const double* dt, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* dt_bias, double* y,
                    double* state_out, double* ckpt) {
  if (!dims_ok(m)) return -1;
  const int NS = m->n_seqs, L = m->n_tok, H = m->n_head, P = m->head_dim, N = m->d_state;
  const int n_chunks = (L + m->chunk - 1) / m->chunk;
  double* hs = (double*)malloc(sizeof(double) * 2 * (size_t)N);
  if (!hs) return -2;
  for (int b = 0; b < NS; b++) {
    const int row = state_row(ids, b);
    if (s0 && (row < 0 || row >= m->state_rows)) { free(hs); return -1; }
    for (int h = 0; h < H; h++)
      for (int p = 0; p < P; p++) {
        double* cur = hs;
        double* nxt = hs + N;
        for (int n = 0; n < N; n++)
          cur[n] = s0 ? s0[(((long)row * H + h) * P + p) * N + n] : 0.0;
        for (int t = 0; t < L; t++) {
          if (ckpt && t % m->chunk == 0) /* state at the START of chunk t / chunk */
            memcpy(ckpt + ((((long)b * n_chunks + t / m->chunk) * H + h) * P + p) * N, cur,
                   sizeof(double) * N);
          double delta = delta_at(m, dt, dt_bias, b, t, h, NULL);
          double ypre = step_fwd(m, b, t, h, p, x, A, B, C, D, delta, cur, nxt);
          long yi = (((long)b * L + t) * H + h) * P + p;
          y[yi] = z ? ypre * silu_d(z[yi]) : ypre;
          double* tmp = cur; cur = nxt; nxt = tmp;
        }
        if (state_out) memcpy(state_out + (((long)b * H + h) * P + p) * N, cur, sizeof(double) * N);
      }
  }
  free(hs);
  return 0;
}

/* Zero every gradient output that is accumulated into. */
static void zero_grads(const oracle_scan_dims* m, double* d_s0, double* d_dt, double* d_A,
                       double* d_B, double* d_C, double* d_D, double* d_dt_bias) {
  const size_t NS = m->n_seqs, L = m->n_tok, H = m->n_head, P = m->head_dim, N = m->d_state,
               G = m->n_group;
  if (d_s0) memset(d_s0, 0, sizeof(double) * (size_t)m->state_rows * H * P * N);
  memset(d_dt, 0, sizeof(double) * NS * L * H);
  memset(d_A, 0, sizeof(double) * H * (m->a_per_state ? N : 1));
  memset(d_B, 0, sizeof(double) * NS * L * G * N);
  memset(d_C, 0, sizeof(double) * NS * L * G * N);
  if (d_D) memset(d_D, 0, sizeof(double) * H * P);
  if (d_dt_bias) memset(d_dt_bias, 0, sizeof(double) * H);
}

/* Reverse walk over tokens t1-1 down to t0 of channel (b, h, p).
 * hist[(t - t0) * N + n] holds h_{t-1} and hist[(t - t0 + 1) * N + n] holds h_t.
 * carry[n] enters as dL/dh_{t1-1} from later tokens and leaves as dL/dh_{t0-1}.
 * Per token (accumulate_token_step_gradients of infotheory model.rs, with the reverse
 * adjoint dh_t = C^T dy_t + a_{t+1} dh_{t+1} of ssm_backward in backprop_ssm.rs):
 *   gy = dy * silu(z)                 dz = dy * y_pre * silu'(z)
 *   dh = gy * C + carry               dC += gy * h_t
 *   dx = gy * D + delta * sum_n dh*B  dB += dh * delta * x
 *   ddelta = sum_n dh * (A * a * h_{t-1} + x * B)
 *   dA += dh * h_{t-1} * a * delta    dD += gy * x      carry = dh * a            */
static void reverse_span(const oracle_scan_dims* m, int b, int h, int p, int t0, int t1,
                         const double* hist, double* carry, const double* x, const double* dt,
                         const double* A, const double* B, const double* C, const double* D,
                         const double* z, const double* dt_bias, const double* dy, double* d_x,
                         double* d_dt, double* d_A, double* d_B, double* d_C, double* d_D,
                         double* d_z, double* d_dt_bias) {
  const int H = m->n_head, P = m->head_dim, N = m->d_state, G = m->n_group, L = m->n_tok;
  const int g = h / (H / G);
  for (int t = t1 - 1; t >= t0; t--) {
    const double* h_prev = hist + (long)(t - t0) * N;
    const double* h_cur = hist + (long)(t - t0 + 1) * N;
    const long yi = (((long)b * L + t) * H + h) * P + p;
    const long bi = (((long)b * L + t) * G + g) * N;
    double pre;
    const double delta = delta_at(m, dt, dt_bias, b, t, h, &pre);
    const double xv = x[yi];
    double ypre = 0.0;
    for (int n = 0; n < N; n++) ypre += C[bi + n] * h_cur[n];
    if (D) ypre += D[h * P + p] * xv;
    double gy = dy[yi];
    if (z) {
      d_z[yi] = dy[yi] * ypre * silu_grad_d(z[yi]);
      gy = dy[yi] * silu_d(z[yi]);
    }
    double sB = 0.0, ddelta = 0.0;
    for (int n = 0; n < N; n++) {
      const double an = a_coef(m, A, h, n);
      const double a = exp(delta * an);
      const double dh = gy * C[bi + n] + carry[n];
      d_C[bi + n] += gy * h_cur[n];
      sB += dh * B[bi + n];
      d_B[bi + n] += dh * delta * xv;
      const double w = dh * h_prev[n] * a;
      ddelta += w * an;
      d_A[m->a_per_state ? (long)h * N + n : h] += w * delta;
      carry[n] = dh * a;
    }
    ddelta += xv * sB;
    d_x[yi] = (D ? gy * D[h * P + p] : 0.0) + delta * sB;
    if (D) d_D[h * P + p] += gy * xv;
    double ddt = m->dt_softplus ? ddelta * softplus_grad_d(pre) : ddelta;
    d_dt[((long)b * L + t) * H + h] += ddt;
    if (m->dt_softplus && d_dt_bias) d_dt_bias[h] += ddt;
  }
}

static int scan_bwd_common(const oracle_scan_dims* m, const double* s0, const double* ckpt,
                           const int* ids, const double* x, const double* dt, const double* A,
                           const double* B, const double* C, const double* D, const double* z,
                           const double* dt_bias, const double* dy, const double* d_state_out,
                           double* d_s0, double* d_x, double* d_dt, double* d_A, double* d_B,
                           double* d_C, double* d_D, double* d_z, double* d_dt_bias) {
  if (!dims_ok(m)) return -1;
  const int NS = m->n_seqs, L = m->n_tok, H = m->n_head, P = m->head_dim, N = m->d_state;
  const int span = ckpt ? m->chunk : L; /* tokens recomputed and held at once */
  const int n_chunks = (L + m->chunk - 1) / m->chunk;
  double* hist = (double*)malloc(sizeof(double) * ((size_t)span + 1) * N);
  double* carry = (double*)malloc(sizeof(double) * (size_t)N);
  if (!hist || !carry) { free(hist); free(carry); return -2; }
  zero_grads(m, d_s0, d_dt, d_A, d_B, d_C, d_D, d_dt_bias);
  for (int b = 0; b < NS; b++) {
    const int row = state_row(ids, b);
    if ((s0 || d_s0) && (row < 0 || row >= m->state_rows)) { free(hist); free(carry); return -1; }
    for (int h = 0; h < H; h++)
      for (int p = 0; p < P; p++) {
        const long sidx = (((long)b * H + h) * P + p) * N;
        for (int n = 0; n < N; n++) carry[n] = d_state_out ? d_state_out[sidx + n] : 0.0;
        const int n_spans = ckpt ? n_chunks : 1;
        for (int s = n_spans - 1; s >= 0; s--) {
          const int t0 = s * span;
          const int t1 = (t0 + span < L) ? t0 + span : L;
          /* start state of the span: the checkpoint (TBPTT replay), or s0 */
          for (int n = 0; n < N; n++) {
            if (ckpt)
              hist[n] = ckpt[((((long)b * n_chunks + s) * H + h) * P + p) * N + n];
            else
              hist[n] = s0 ? s0[(((long)row * H + h) * P + p) * N + n] : 0.0;
          }
          for (int t = t0; t < t1; t++) {
            double delta = delta_at(m, dt, dt_bias, b, t, h, NULL);
            step_fwd(m, b, t, h, p, x, A, B, C, D, delta, hist + (long)(t - t0) * N,
                     hist + (long)(t - t0 + 1) * N);
          }
          reverse_span(m, b, h, p, t0, t1, hist, carry, x, dt, A, B, C, D, z, dt_bias, dy, d_x,
                       d_dt, d_A, d_B, d_C, d_D, d_z, d_dt_bias);
        }
        /* dL/dh_{-1} = a_0 * dh_0 (ssm_backward: grad_hidden_init), summed per state row */
        if (d_s0)
          for (int n = 0; n < N; n++) d_s0[(((long)row * H + h) * P + p) * N + n] += carry[n];
      }
  }
  free(hist);
  free(carry);
  return 0;
}

int oracle_scan_bwd(const oracle_scan_dims* m, const double* s0, const int* ids, const double* x,
                    const double* dt, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* dt_bias, const double* dy,
                    const double* d_state_out, double* d_s0, double* d_x, double* d_dt,
                    double* d_A, double* d_B, double* d_C, double* d_D, double* d_z,
                    double* d_dt_bias) {
  return scan_bwd_common(m, s0, NULL, ids, x, dt, A, B, C, D, z, dt_bias, dy, d_state_out, d_s0,
                         d_x, d_dt, d_A, d_B, d_C, d_D, d_z, d_dt_bias);
}

int oracle_scan_bwd_ckpt(const oracle_scan_dims* m, const double* ckpt, const int* ids,
                         const double* x, const double* dt, const double* A, const double* B,
                         const double* C, const double* D, const double* z, const double* dt_bias,
                         const double* dy, const double* d_state_out, double* d_s0, double* d_x,
                         double* d_dt, double* d_A, double* d_B, double* d_C, double* d_D,
                         double* d_z, double* d_dt_bias) {
  if (!ckpt) return -1;
  return scan_bwd_common(m, NULL, ckpt, ids, x, dt, A, B, C, D, z, dt_bias, dy, d_state_out, d_s0,
                         d_x, d_dt, d_A, d_B, d_C, d_D, d_z, d_dt_bias);
}

/* ---- states by balanced-tree composition ------------------------------------------
 * The step h_t = a_t h_{t-1} + u_t is the affine map (a_t, u_t).  Applying (a1, u1) then
 * (a2, u2) is (a2 a1, a2 u1 + u2), an associative operator (associative_scan_backward of
 * backprop_ssm.rs scans exactly this recurrence).  Here the inclusive prefix over [lo, hi)
 * is built by splitting the range in halves, scanning each half on its own and composing
 * the left total into every element of the right half. */
static void tree_prefix(double* a, double* u, int lo, int hi) {
  if (hi - lo <= 1) return;
  int mid = lo + (hi - lo) / 2;
  tree_prefix(a, u, lo, mid);
  tree_prefix(a, u, mid, hi);
  const double la = a[mid - 1], lu = u[mid - 1];
  for (int i = mid; i < hi; i++) { /* (la, lu) first, then the right-half prefix */
    u[i] = a[i] * lu + u[i];
    a[i] = a[i] * la;
  }
}

int oracle_scan_states_assoc(const oracle_scan_dims* m, const double* s0, const int* ids,
                             const double* x, const double* dt, const double* A, const double* B,
                             const double* dt_bias, double* states) {
  if (!dims_ok(m)) return -1;
  const int NS = m->n_seqs, L = m->n_tok, H = m->n_head, P = m->head_dim, N = m->d_state,
            G = m->n_group;
  double* a = (double*)malloc(sizeof(double) * (size_t)L);
  double* u = (double*)malloc(sizeof(double) * (size_t)L);
  if (!a || !u) { free(a); free(u); return -2; }
  for (int b = 0; b < NS; b++) {
    const int row = state_row(ids, b);
    for (int h = 0; h < H; h++) {
      const int g = h / (H / G);
      for (int p = 0; p < P; p++)
        for (int n = 0; n < N; n++) {
          for (int t = 0; t < L; t++) {
            double delta = delta_at(m, dt, dt_bias, b, t, h, NULL);
            double xv = x[(((long)b * L + t) * H + h) * P + p];
            a[t] = exp(delta * a_coef(m, A, h, n));
            u[t] = delta * xv * B[(((long)b * L + t) * G + g) * N + n];
          }
          tree_prefix(a, u, 0, L);
          double h0 = s0 ? s0[(((long)row * H + h) * P + p) * N + n] : 0.0;
          for (int t = 0; t < L; t++)
            states[((((long)b * L + t) * H + h) * P + p) * N + n] = a[t] * h0 + u[t];
        }
    }
  }
  free(a);
  free(u);
  return 0;
}
