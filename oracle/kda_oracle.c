/*
 * kda_oracle.c -- plain CPU oracle for the fused causal-conv1d + KDA
 * (gated delta-rule) multi-token-prediction verify decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant generator with the
 * CUDA library.
 *
 * Source of the definition: "[KDA] Fuse causal conv1d into MTP verify
 * decode" (cuLA pull request 107), its description section and its two
 * commit messages.  The op consumes packed pre-convolution mixed_qkv and
 * performs, per sequence and value head: a width-W depthwise causal conv1d
 * over [conv_state || T new tokens] followed by SiLU (applied to the q, k and
 * v channels, the "v-conv"), q/k L2 normalisation, the gate and beta, and the
 * gated delta-rule recurrence
 *
 *     S <- diag(exp g) S
 *     S <- S + beta k (v - S^T k)^T
 *     o  = K^{-1/2} S^T q
 *
 * token by token, with the persistent state read-only, a snapshot of S after
 * every token, a snapshot of the raw conv window after every token, and
 * conv_state rolled to the last W-1 raw inputs.  The softplus gate follows
 * the review thread on the same page: a real branch, linear above the
 * threshold, so an overflowing exp is never evaluated.
 *
 * Everything is double precision, written as the definition reads: no
 * blocking, fusion or reordering.  Readings of points the page leaves open
 * (channel order, tap order, no conv bias, L2-norm epsilon, snapshot
 * contents, GVA head map) are stated next to the code that takes them.
 *
 * Build:  gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared kda_oracle.c -lm
 * (-ffp-contract=off keeps a*b+c unfused so x86 and Arm hosts agree.)
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EBADARG -1
#define ORC_ENOMEM -2

#define ORC_GATE_SOFTPLUS 0
#define ORC_GATE_SAFE 1

/* ---- scalar functions ---------------------------------------------------- */

/* SiLU(y) = y * sigmoid(y). */
double orc_silu(double y) { return y / (1.0 + exp(-y)); }

/* beta = sigmoid(b). */
double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus with beta_sp = 1 and threshold 20: identity above the threshold,
 * log(1 + e^x) otherwise.  A true branch (review thread of the PR page): the
 * exponential is only evaluated where it cannot overflow. */
double orc_softplus(double x) {
  if (x > 20.0) return x;
  return log1p(exp(x));
}

/* Softplus gate: g = -exp(A_log) * softplus(a + dt_bias). */
double orc_gate_softplus(double A_log, double a, double dt_bias) {
  return -exp(A_log) * orc_softplus(a + dt_bias);
}

/* Safe gate: the input already is the log-decay; it is clamped to <= 0. */
double orc_gate_safe(double a) { return a < 0.0 ? a : 0.0; }

/* ---- step functions ------------------------------------------------------ */

/* Causal depthwise conv of one channel.
 * xext holds the W-1 state values (oldest first) followed by the T new raw
 * inputs; tap W-1 multiplies the newest input of each window (the usual
 * causal-conv1d convention; the page does not spell it out).  No bias.
 * y[t] = silu( sum_{j=0}^{W-1} w[j] * xext[t+j] ). */
void orc_causal_conv1d_silu(int T, int W, const double* xext, const double* w,
                            double* y) {
  for (int t = 0; t < T; ++t) {
    double acc = 0.0;
    for (int j = 0; j < W; ++j) acc += w[j] * xext[t + j];
    y[t] = orc_silu(acc);
  }
}

/* x <- x / sqrt(sum x^2 + eps).  The page says "L2 normalization" without an
 * epsilon; eps sits inside the square root (the common l2norm kernel form). */
void orc_l2norm(int n, double* x, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) x[i] *= inv;
}

/* One token of the gated delta rule on a K x V state (row k, column v, v
 * contiguous).  g[K] is the channel-wise log-decay, k/q already
 * L2-normalised, scale = K^{-1/2}.  Writes o[V]; S is updated in place. */
void orc_delta_rule_step(int K, int V, double* S, const double* g,
                         const double* k, const double* v, double beta,
                         const double* q, double scale, double* o) {
  /* S <- diag(exp g) S */
  for (int r = 0; r < K; ++r) {
    double d = exp(g[r]);
    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] *= d;
  }
  /* S <- S + beta k (v - S^T k)^T */
  double* u = (double*)malloc(sizeof(double) * (size_t)V);
  for (int c = 0; c < V; ++c) {
    double sk = 0.0;
    for (int r = 0; r < K; ++r) sk += S[(size_t)r * V + c] * k[r];
    u[c] = v[c] - sk;
  }
  for (int r = 0; r < K; ++r)
    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] += beta * k[r] * u[c];
  free(u);
  /* o = K^{-1/2} S^T q */
  for (int c = 0; c < V; ++c) {
    double sq = 0.0;
    for (int r = 0; r < K; ++r) sq += S[(size_t)r * V + c] * q[r];
    o[c] = scale * sq;
  }
}

/* ---- one sequence -------------------------------------------------------- */

/* The whole verify call for ONE sequence (all heads).  Layouts, dense:
 *   x       [T][dim]        this sequence's mixed_qkv; dim = 2HK + HV V;
 *                           channels q (H heads of K) | k (H x K) | v (HV x V)
 *   w       [dim][W]        conv weights
 *   cs      [dim][W-1]      conv_state before the call, oldest first
 *   A_log   [HV], dt_bias [HV][K]   softplus gate only (may be NULL for safe)
 *   a       [T][HV][K]      gate input (safe gate: the log-decay itself)
 *   b       [T][HV]         beta logit
 *   S0      [HV][K][V]      persistent state, read only
 * Outputs:
 *   o       [T][HV][V]
 *   inter   [T][HV][K][V]   S after token t
 *   snap    [T][dim][W-1]   raw conv window after accepting token t: the
 *                           W-1 newest raw inputs, i.e. xext[t+1 .. t+W-1]
 *                           (the state a rollback to token t restores)
 *   cs_new  [dim][W-1]      conv_state after the call = xext[T .. T+W-2]
 * Value head hv reads q/k head hv / (HV/H) (consecutive grouping).
 */
int orc_kda_conv_verify_seq(int T, int H, int HV, int K, int V, int W,
                            int gate_mode, double eps, const double* x,
                            const double* w, const double* cs,
                            const double* A_log, const double* dt_bias,
                            const double* a, const double* b, const double* S0,
                            double* o, double* inter, double* snap,
                            double* cs_new) {
  if (T < 1 || H < 1 || HV < H || HV % H != 0 || K < 1 || V < 1 || W < 1)
    return ORC_EBADARG;
  if (gate_mode == ORC_GATE_SOFTPLUS && (!A_log || !dt_bias)) return ORC_EBADARG;
  if (gate_mode != ORC_GATE_SOFTPLUS && gate_mode != ORC_GATE_SAFE)
    return ORC_EBADARG;
  const int dim = 2 * H * K + HV * V;
  const int G = HV / H;
  const int L = T + W - 1;

  double* y = (double*)malloc(sizeof(double) * (size_t)T * dim);
  double* xext = (double*)malloc(sizeof(double) * (size_t)L);
  double* yc = (double*)malloc(sizeof(double) * (size_t)T);
  double* S = (double*)malloc(sizeof(double) * (size_t)K * V);
  double* qn = (double*)malloc(sizeof(double) * (size_t)K);
  double* kn = (double*)malloc(sizeof(double) * (size_t)K);
  double* g = (double*)malloc(sizeof(double) * (size_t)K);
  if (!y || !xext || !yc || !S || !qn || !kn || !g) {
    free(y); free(xext); free(yc); free(S); free(qn); free(kn); free(g);
    return ORC_ENOMEM;
  }

  /* Conv + SiLU on every channel, conv-window snapshots, conv_state roll. */
  for (int c = 0; c < dim; ++c) {
    for (int j = 0; j < W - 1; ++j) xext[j] = cs[(size_t)c * (W - 1) + j];
    for (int t = 0; t < T; ++t) xext[W - 1 + t] = x[(size_t)t * dim + c];
    orc_causal_conv1d_silu(T, W, xext, w + (size_t)c * W, yc);
    for (int t = 0; t < T; ++t) y[(size_t)t * dim + c] = yc[t];
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < W - 1; ++j)
        snap[((size_t)t * dim + c) * (W - 1) + j] = xext[t + 1 + j];
    for (int j = 0; j < W - 1; ++j) cs_new[(size_t)c * (W - 1) + j] = xext[T + j];
  }

  const double scale = 1.0 / sqrt((double)K);
  for (int hv = 0; hv < HV; ++hv) {
    const int h = hv / G;
    memcpy(S, S0 + (size_t)hv * K * V, sizeof(double) * (size_t)K * V);
    for (int t = 0; t < T; ++t) {
      const double* yt = y + (size_t)t * dim;
      for (int r = 0; r < K; ++r) {
        qn[r] = yt[h * K + r];
        kn[r] = yt[H * K + h * K + r];
      }
      orc_l2norm(K, qn, eps);
      orc_l2norm(K, kn, eps);
      const double* vt = yt + 2 * H * K + hv * V;
      const double* at = a + ((size_t)t * HV + hv) * K;
      for (int r = 0; r < K; ++r)
        g[r] = gate_mode == ORC_GATE_SOFTPLUS
                   ? orc_gate_softplus(A_log[hv], at[r], dt_bias[(size_t)hv * K + r])
                   : orc_gate_safe(at[r]);
      const double beta = orc_sigmoid(b[(size_t)t * HV + hv]);
      orc_delta_rule_step(K, V, S, g, kn, vt, beta, qn, scale,
                          o + ((size_t)t * HV + hv) * V);
      memcpy(inter + ((size_t)t * HV + hv) * K * V, S, sizeof(double) * (size_t)K * V);
    }
  }
  free(y); free(xext); free(yc); free(S); free(qn); free(kn); free(g);
  return ORC_OK;
}

/* ---- commit after verify ------------------------------------------------- */

/* Accept the first `acc` (1 <= acc <= T) verified tokens of ONE sequence:
 * the persistent state becomes the state snapshot after token acc-1 and the
 * conv_state becomes the conv-window snapshot after token acc-1 (the rollback
 * the per-token snapshots exist for, per the verify-decode page).
 *   inter   [T][HV][K][V],  snap [T][dim][W-1]  (this sequence's snapshots)
 *   S_out   [HV][K][V],     cs_out [dim][W-1]
 * Returns ORC_EBADARG (and writes nothing) when acc is out of range. */
int orc_commit_seq(int T, int HV, int K, int V, int dim, int W, int acc, const double* inter,
                   const double* snap, double* S_out, double* cs_out) {
  if (acc < 1 || acc > T) return ORC_EBADARG;
  const size_t ns = (size_t)HV * K * V, nc = (size_t)dim * (W - 1);
  memcpy(S_out, inter + (size_t)(acc - 1) * ns, sizeof(double) * ns);
  memcpy(cs_out, snap + (size_t)(acc - 1) * nc, sizeof(double) * nc);
  return ORC_OK;
}
