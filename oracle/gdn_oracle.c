/*
 * gdn_oracle.c -- plain, slow, sequential fp64 CPU reference of the Gated
 * DeltaNet (GDN) layer hot path.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or helper with
 * the CUDA library; neither includes nor links the other.
 *
 * What it computes (sources by page title and section):
 *   [P1] RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv
 *        state contract":
 *        - Summary, conv bullet: the conv accumulator is fp32, starts from the
 *          bias, and each tap product is rounded to the operand dtype before
 *          it is added.
 *        - Summary, provider bullet + Notes "How the golden relates to the
 *          kernel": fused fp32 gating beta = sigmoid(b), g = -exp(A_log) *
 *          softplus(a + dt_bias) with the softplus threshold at 20; the QK
 *          norm x / sqrt(sum(x*x) + 1e-6) with scale on q after the norm;
 *          k-head of value head h is h / (HV / H).
 *        - Summary, state ABI bullet + Notes "State ABI": recurrent state
 *          [num_blocks, HV, V, K]; conv state [num_blocks, dim, W-1] or the
 *          transposed layout; slots <= 0 are skipped (zero output, state
 *          untouched); the goldens reject out-of-range or repeated slots.
 *   The recurrence itself (the gated delta rule that GatedDeltaRuleRecurrent-
 *   StepOp of [P1] implements): per value head,
 *        S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) k_t^T,  o_t = S_t q_t,
 *   taken in the order decay -> predict -> correct -> read out.
 *   [P4] vLLM PR #53864 "Numerical root cause and fix": the chunked prefill
 *        inverts the lower-triangular per-chunk KK^T block; three
 *        Newton-Schulz rounds with bf16 intermediates fail on correlated keys.
 *   [P1] page, Summary by CodeRabbit and Walkthrough (RL-Kernel PRs #466-#468,
 *        "Gated RMSNorm CUDA kernel for the GDN block"): the GDN output goes
 *        through a gated RMSNorm, with SiLU or sigmoid gating and a weight
 *        offset (zero for the plain form, one for the zero-centred one).
 *
 * Precision: everything is fp64 except where [P1] fixes it -- the conv
 * accumulator (fp32, each add rounded to fp32) and the tap products (rounded
 * to the operand dtype). Outputs are returned unrounded in fp64 and, where the
 * layer's output is bf16, also rounded once (round-to-nearest-even) to bf16.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fPIC -shared gdn_oracle.c -lm -lpthread
 * (-ffp-contract=off: no fused multiply-add may merge a rounded product into
 * the following add).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 / fp32 conversions (IEEE 754 definitions)                            */
/* ------------------------------------------------------------------------ */

/* bf16 bits -> value (exact: bf16 is the top half of a binary32). */
static double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static uint16_t f32_bits_hi(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* One rounding of a double to bf16 (8 significant bits, binary32 exponent
 * range, subnormal quantum 2^-133), ties to even. */
uint16_t gdn_ref_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double ax = fabs(x);
  if (ax == 0.0) return sign;
  if (isinf(ax)) return sign | 0x7F80;
  int e;
  frexp(ax, &e);           /* ax = m * 2^e, m in [0.5, 1) */
  int qexp = e - 8;        /* quantum of an 8-significant-bit number in [2^(e-1), 2^e) */
  if (qexp < -133) qexp = -133;
  double r = ldexp(nearbyint(ldexp(ax, -qexp)), qexp); /* nearbyint: ties to even */
  if (r >= 0x1p128) return sign | 0x7F80;               /* beyond the largest finite bf16 */
  return sign | f32_bits_hi((float)r);                  /* r is exact in binary32 */
}

static double round_bf16_val(double x) { return bf16_to_f64(gdn_ref_round_bf16(x)); }

/* binary32 add / multiply from exact-or-wider fp64 operations: fp64 has more
 * than 2*24+2 significant bits, so rounding the fp64 result once more to
 * binary32 gives the correctly rounded binary32 result. */
static float f32_add(float a, float b) { return (float)((double)a + (double)b); }

/* ------------------------------------------------------------------------ */
/* Conv state pool access                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  void* base;   /* pool base */
  int f32;      /* 1: binary32 entries, 0: bf16 entries */
  int layout;   /* 0: [slots, D, W-1], 1: [slots, W-1, D] */
  int D, W;
} conv_pool;

static size_t conv_index(const conv_pool* p, int slot, int c, int j) {
  if (p->layout == 0) return ((size_t)slot * p->D + c) * (size_t)(p->W - 1) + j;
  return ((size_t)slot * (p->W - 1) + j) * (size_t)p->D + c;
}

static double conv_get(const conv_pool* p, int slot, int c, int j) {
  size_t i = conv_index(p, slot, c, j);
  if (p->f32) return (double)((const float*)p->base)[i];
  return bf16_to_f64(((const uint16_t*)p->base)[i]);
}

/* Stores a value that is exactly representable in the pool's dtype. */
static void conv_put(const conv_pool* p, int slot, int c, int j, double v) {
  size_t i = conv_index(p, slot, c, j);
  if (p->f32) ((float*)p->base)[i] = (float)v;
  else ((uint16_t*)p->base)[i] = gdn_ref_round_bf16(v);
}

/* ------------------------------------------------------------------------ */
/* One conv output ([P1] Summary, conv bullet)                               */
/* ------------------------------------------------------------------------ */

/* win[0..W-1]: the W window values, oldest first (win[W-1] = newest input).
 * w[0..W-1]: the channel's taps. Returns the fp32 pre-activation and writes
 * the bf16 output bits. */
static float conv_channel(const double* win, const uint16_t* w, const uint16_t* bias_c,
                          int W, int cache_f32, int silu, uint16_t* out_bits, double* out_act) {
  float acc = bias_c ? (float)bf16_to_f64(*bias_c) : 0.0f;
  for (int j = 0; j < W; ++j) {
    double p = bf16_to_f64(w[j]) * win[j]; /* exact: <= 8 x 24 significant bits */
    float pr = cache_f32 ? (float)p : (float)round_bf16_val(p);
    acc = f32_add(acc, pr);
  }
  double y = (double)acc;
  if (silu) y = y / (1.0 + exp(-y));
  if (out_act) *out_act = y;
  *out_bits = gdn_ref_round_bf16(y);
  return acc;
}

/* Conv of every channel of one row / token against a window pool held in
 * `win` ([D][W-1] doubles, oldest first); rolls `win` by one. */
static void conv_row(double* win, const uint16_t* x, const uint16_t* weight, const uint16_t* bias,
                     int D, int W, int cache_f32, int silu, uint16_t* y_bits, double* y_act) {
  double full[16];
  for (int c = 0; c < D; ++c) {
    for (int j = 0; j < W - 1; ++j) full[j] = win[(size_t)c * (W - 1) + j];
    full[W - 1] = bf16_to_f64(x[c]);
    conv_channel(full, weight + (size_t)c * W, bias ? bias + c : NULL, W, cache_f32, silu,
                 &y_bits[c], y_act ? &y_act[c] : NULL);
    for (int j = 0; j < W - 1; ++j) win[(size_t)c * (W - 1) + j] = full[j + 1];
  }
}

/* ------------------------------------------------------------------------ */
/* Gating and QK norm ([P1] Notes, "How the golden relates to the kernel")   */
/* ------------------------------------------------------------------------ */

double gdn_ref_softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }
double gdn_ref_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* gate_direct = 0: a, b are bf16 bits; g = -exp(A_log) softplus(a + dt_bias),
 * beta = sigmoid(b). gate_direct = 1: a, b are binary32 g and beta. */
static void gate_values(const void* a, const void* b, int gate_direct, const float* A_log,
                        const float* dt_bias, size_t idx, int h, double* g, double* beta) {
  if (gate_direct) {
    *g = (double)((const float*)a)[idx];
    *beta = (double)((const float*)b)[idx];
  } else {
    double av = bf16_to_f64(((const uint16_t*)a)[idx]);
    double bv = bf16_to_f64(((const uint16_t*)b)[idx]);
    *g = -exp((double)A_log[h]) * gdn_ref_softplus(av + (double)dt_bias[h]);
    *beta = gdn_ref_sigmoid(bv);
  }
}

/* x <- x / sqrt(sum x^2 + 1e-6) (if l2norm), then x <- x * mult. */
static void qk_normalise(double* x, int n, int l2norm, double mult) {
  double inv = 1.0;
  if (l2norm) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    inv = 1.0 / sqrt(ss + 1e-6);
  }
  for (int i = 0; i < n; ++i) x[i] = x[i] * inv * mult;
}

/* ------------------------------------------------------------------------ */
/* The gated delta rule, one head, one token                                 */
/* ------------------------------------------------------------------------ */

/* S: [dv][dk]. q, k: [dk] (already normalised / scaled). v: [dv]. o: [dv]. */
static void delta_rule_token(double* S, const double* q, const double* k, const double* v,
                             double g, double beta, int dk, int dv, double* o) {
  double alpha = exp(g);
  for (int r = 0; r < dv; ++r) {
    double* Sr = S + (size_t)r * dk;
    for (int c = 0; c < dk; ++c) Sr[c] *= alpha;         /* decay */
    double pred = 0.0;
    for (int c = 0; c < dk; ++c) pred += Sr[c] * k[c];   /* predict: (a S) k */
    double delta = beta * (v[r] - pred);                 /* correct */
    for (int c = 0; c < dk; ++c) Sr[c] += delta * k[c];  /* rank-1 update */
    double out = 0.0;
    for (int c = 0; c < dk; ++c) out += Sr[c] * q[c];    /* read out */
    o[r] = out;
  }
}

/* Token-by-token recurrence for one head over T tokens.
 * q, k: [T][dk]; v: [T][dv]; g, beta: [T]; S: [dv][dk] in/out; o: [T][dv]. */
void gdn_ref_recurrent_head(const double* q, const double* k, const double* v, const double* g,
                            const double* beta, double* S, int T, int dk, int dv, double* o) {
  for (int t = 0; t < T; ++t)
    delta_rule_token(S, q + (size_t)t * dk, k + (size_t)t * dk, v + (size_t)t * dv, g[t],
                     beta[t], dk, dv, o + (size_t)t * dv);
}

/* ------------------------------------------------------------------------ */
/* The chunked (UT / WY) form, one head -- a second fp64 path                */
/* ------------------------------------------------------------------------ */
/*
 * Within a chunk that starts from state S0, with G_t the running sum of g
 * inside the chunk (inclusive) and gamma_t = exp(G_t), unrolling the rule
 * gives S_t = gamma_t S0 + sum_{j<=t} (gamma_t/gamma_j) d_j k_j^T, where the
 * corrections d_j solve the unit lower-triangular system
 *   (I + A) D = diag(beta) V - diag(beta gamma) K S0^T,
 *   A_tj = beta_t exp(G_t - G_j) (k_t . k_j)  for j < t.
 * With T = (I + A)^-1:  U = T diag(beta) V,  W = T diag(beta gamma) K,
 *   D = U - W S0^T,
 *   O = diag(gamma) Q S0^T + (M o Q K^T) D,   M_tj = exp(G_t - G_j), j <= t,
 *   S_end = gamma_last S0 + D^T diag(exp(G_last - G_j)) K.
 * ([P4] "Numerical root cause and fix" names the per-chunk KK^T block and its
 * lower-triangular inverse; the algebra above is derived from the rule.)
 */

/* Exact inverse of the unit lower-triangular n x n matrix I + A (A strictly
 * lower, row-major) by forward substitution, column by column. */
void gdn_ref_unit_lower_inverse(const double* A, int n, double* T) {
  for (int col = 0; col < n; ++col) {
    for (int r = 0; r < n; ++r) {
      double s = (r == col) ? 1.0 : 0.0;
      for (int j = col; j < r; ++j) s -= A[(size_t)r * n + j] * T[(size_t)j * n + col];
      T[(size_t)r * n + col] = (r < col) ? 0.0 : s;
    }
  }
}

/* The approximation the [P4] page replaces: inverse of each 16x16 diagonal
 * block of M = I + A by `rounds` Newton-Schulz steps X <- X (2I - M X) from
 * X0 = I - A_block, with every intermediate matrix rounded to bf16; the
 * off-diagonal blocks then follow exactly (fp64) by block forward
 * substitution from those diagonal inverses. Used only as a negative control. */
static void ns_bf16_block_inverse(const double* A, int n, int rounds, double* T) {
  enum { NB = 16 };
  double M[NB * NB], X[NB * NB], MX[NB * NB], Y[NB * NB];
  double* Dinv = (double*)calloc((size_t)n * n, sizeof(double));
  for (int b0 = 0; b0 < n; b0 += NB) {
    int nb = (n - b0 < NB) ? n - b0 : NB;
    for (int i = 0; i < nb; ++i)
      for (int j = 0; j < nb; ++j) {
        double a = (j < i) ? A[(size_t)(b0 + i) * n + (b0 + j)] : 0.0;
        M[i * NB + j] = round_bf16_val((i == j ? 1.0 : 0.0) + a);
        X[i * NB + j] = round_bf16_val((i == j ? 1.0 : 0.0) - a);
      }
    for (int it = 0; it < rounds; ++it) {
      for (int i = 0; i < nb; ++i)
        for (int j = 0; j < nb; ++j) {
          double s = 0.0;
          for (int l = 0; l < nb; ++l) s += M[i * NB + l] * X[l * NB + j];
          MX[i * NB + j] = round_bf16_val(((i == j) ? 2.0 : 0.0) - s);
        }
      for (int i = 0; i < nb; ++i)
        for (int j = 0; j < nb; ++j) {
          double s = 0.0;
          for (int l = 0; l < nb; ++l) s += X[i * NB + l] * MX[l * NB + j];
          Y[i * NB + j] = round_bf16_val(s);
        }
      memcpy(X, Y, sizeof X);
    }
    for (int i = 0; i < nb; ++i)
      for (int j = 0; j < nb; ++j) Dinv[(size_t)(b0 + i) * n + (b0 + j)] = X[i * NB + j];
  }
  /* block forward substitution: T_rc = -Dinv_r sum_{c <= l < r} A_rl T_lc */
  memset(T, 0, (size_t)n * n * sizeof(double));
  for (int r0 = 0; r0 < n; r0 += NB) {
    int nr = (n - r0 < NB) ? n - r0 : NB;
    for (int i = 0; i < nr; ++i)
      for (int j = 0; j < nr; ++j)
        T[(size_t)(r0 + i) * n + (r0 + j)] = Dinv[(size_t)(r0 + i) * n + (r0 + j)];
    for (int c0 = 0; c0 < r0; c0 += NB) {
      int nc = (n - c0 < NB) ? n - c0 : NB;
      for (int i = 0; i < nr; ++i)
        for (int j = 0; j < nc; ++j) {
          double acc = 0.0; /* (sum_l A_rl T_lc)_(i,j) over l in [c0, r0) */
          for (int l = c0; l < r0; ++l)
            acc += A[(size_t)(r0 + i) * n + l] * T[(size_t)l * n + (c0 + j)];
          Y[i * NB + j] = acc;
        }
      for (int i = 0; i < nr; ++i)
        for (int j = 0; j < nc; ++j) {
          double acc = 0.0;
          for (int l = 0; l < nr; ++l)
            acc += Dinv[(size_t)(r0 + i) * n + (r0 + l)] * Y[l * NB + j];
          T[(size_t)(r0 + i) * n + (c0 + j)] = -acc;
        }
    }
  }
  free(Dinv);
}

/* Chunked form for one head. inverse_mode: 0 = exact forward substitution;
 * k > 0 = the bf16 Newton-Schulz block inverse with k rounds (negative
 * control). Arguments as gdn_ref_recurrent_head, plus chunk size C. */
void gdn_ref_chunked_head(const double* q, const double* k, const double* v, const double* g,
                          const double* beta, double* S, int T, int dk, int dv, int C,
                          int inverse_mode, double* o) {
  double* G = (double*)malloc(sizeof(double) * C);
  double* A = (double*)malloc(sizeof(double) * C * C);
  double* Tinv = (double*)malloc(sizeof(double) * C * C);
  double* U = (double*)malloc(sizeof(double) * C * dv);
  double* Wm = (double*)malloc(sizeof(double) * C * dk);
  double* Dl = (double*)malloc(sizeof(double) * C * dv);
  double* Snew = (double*)malloc(sizeof(double) * dv * dk);
  for (int t0 = 0; t0 < T; t0 += C) {
    int L = (T - t0 < C) ? T - t0 : C;
    const double* Q = q + (size_t)t0 * dk;
    const double* K = k + (size_t)t0 * dk;
    const double* V = v + (size_t)t0 * dv;
    const double* bt = beta + t0;
    double run = 0.0;
    for (int t = 0; t < L; ++t) { run += g[t0 + t]; G[t] = run; }
    /* A_tj = beta_t exp(G_t - G_j) k_t . k_j, j < t */
    for (int t = 0; t < L; ++t)
      for (int j = 0; j < L; ++j) {
        double a = 0.0;
        if (j < t) {
          double kk = 0.0;
          for (int c = 0; c < dk; ++c) kk += K[(size_t)t * dk + c] * K[(size_t)j * dk + c];
          a = bt[t] * exp(G[t] - G[j]) * kk;
        }
        A[t * L + j] = a;
      }
    if (inverse_mode == 0) gdn_ref_unit_lower_inverse(A, L, Tinv);
    else ns_bf16_block_inverse(A, L, inverse_mode, Tinv);
    /* U = T diag(beta) V ; W = T diag(beta gamma) K */
    for (int t = 0; t < L; ++t) {
      for (int r = 0; r < dv; ++r) {
        double s = 0.0;
        for (int j = 0; j < L; ++j) s += Tinv[t * L + j] * bt[j] * V[(size_t)j * dv + r];
        U[(size_t)t * dv + r] = s;
      }
      for (int c = 0; c < dk; ++c) {
        double s = 0.0;
        for (int j = 0; j < L; ++j) s += Tinv[t * L + j] * bt[j] * exp(G[j]) * K[(size_t)j * dk + c];
        Wm[(size_t)t * dk + c] = s;
      }
    }
    /* D = U - W S0^T */
    for (int t = 0; t < L; ++t)
      for (int r = 0; r < dv; ++r) {
        double s = 0.0;
        for (int c = 0; c < dk; ++c) s += Wm[(size_t)t * dk + c] * S[(size_t)r * dk + c];
        Dl[(size_t)t * dv + r] = U[(size_t)t * dv + r] - s;
      }
    /* O = diag(gamma) Q S0^T + (M o Q K^T) D */
    for (int t = 0; t < L; ++t)
      for (int r = 0; r < dv; ++r) {
        double s0 = 0.0;
        for (int c = 0; c < dk; ++c) s0 += Q[(size_t)t * dk + c] * S[(size_t)r * dk + c];
        double s1 = 0.0;
        for (int j = 0; j <= t; ++j) {
          double qk = 0.0;
          for (int c = 0; c < dk; ++c) qk += Q[(size_t)t * dk + c] * K[(size_t)j * dk + c];
          s1 += exp(G[t] - G[j]) * qk * Dl[(size_t)j * dv + r];
        }
        o[(size_t)(t0 + t) * dv + r] = exp(G[t]) * s0 + s1;
      }
    /* S_end = gamma_last S0 + D^T diag(exp(G_last - G_j)) K */
    for (int r = 0; r < dv; ++r)
      for (int c = 0; c < dk; ++c) {
        double s = exp(G[L - 1]) * S[(size_t)r * dk + c];
        for (int j = 0; j < L; ++j)
          s += Dl[(size_t)j * dv + r] * exp(G[L - 1] - G[j]) * K[(size_t)j * dk + c];
        Snew[(size_t)r * dk + c] = s;
      }
    memcpy(S, Snew, sizeof(double) * dv * dk);
  }
  free(G); free(A); free(Tinv); free(U); free(Wm); free(Dl); free(Snew);
}

/* ------------------------------------------------------------------------ */
/* Slot contract ([P1] Notes, "State ABI")                                   */
/* ------------------------------------------------------------------------ */

/* 0: inactive (skip, zero output); 1: active; -1: out of range (error, skip). */
static int slot_class(int32_t s, int num_slots) {
  if (s <= 0) return 0;
  if (s >= num_slots) return -1;
  return 1;
}

int gdn_ref_validate_slots(const int32_t* slot, int n, int num_slots) {
  for (int i = 0; i < n; ++i)
    if (slot[i] > 0 && slot[i] >= num_slots) return 1;
  for (int i = 0; i < n; ++i)
    for (int j = i + 1; j < n; ++j)
      if (slot[i] > 0 && slot[i] == slot[j]) return 2;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Conv update (decode)                                                      */
/* ------------------------------------------------------------------------ */

/* x [B, D] bf16; conv_state pool (cache_f32 ? binary32 : bf16), layout 0/1;
 * weight [D, W] bf16; bias [D] bf16 or NULL; out_bits [B, D] bf16;
 * out_act [B, D] fp64 activation before bf16 rounding (nullable). */
int gdn_ref_conv_update(const uint16_t* x, void* conv_state, int cache_f32, int layout,
                        const uint16_t* weight, const uint16_t* bias, int silu,
                        const int32_t* slot, int B, int D, int W, int num_slots,
                        uint16_t* out_bits, double* out_act, int32_t* err) {
  conv_pool pool = {conv_state, cache_f32, layout, D, W};
  double* win = (double*)malloc(sizeof(double) * (size_t)D * (W - 1));
  for (int b = 0; b < B; ++b) {
    int cls = slot_class(slot[b], num_slots);
    if (cls < 0 && err) *err |= 1;
    if (cls <= 0) {
      memset(out_bits + (size_t)b * D, 0, sizeof(uint16_t) * D);
      if (out_act) memset(out_act + (size_t)b * D, 0, sizeof(double) * D);
      continue;
    }
    int s = slot[b];
    for (int c = 0; c < D; ++c)
      for (int j = 0; j < W - 1; ++j) win[(size_t)c * (W - 1) + j] = conv_get(&pool, s, c, j);
    conv_row(win, x + (size_t)b * D, weight, bias, D, W, cache_f32, silu,
             out_bits + (size_t)b * D, out_act ? out_act + (size_t)b * D : NULL);
    for (int c = 0; c < D; ++c)
      for (int j = 0; j < W - 1; ++j) conv_put(&pool, s, c, j, win[(size_t)c * (W - 1) + j]);
  }
  free(win);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Thread helper: run fn(ctx, unit) for unit in [0, n) over nthreads threads */
/* ------------------------------------------------------------------------ */

typedef void (*unit_fn)(void* ctx, int unit);
typedef struct { unit_fn fn; void* ctx; int n, stride, first; } unit_job;

static void* unit_worker(void* p) {
  unit_job* j = (unit_job*)p;
  for (int u = j->first; u < j->n; u += j->stride) j->fn(j->ctx, u);
  return NULL;
}

static void run_units(unit_fn fn, void* ctx, int n, int nthreads) {
  if (nthreads <= 1 || n <= 1) {
    for (int u = 0; u < n; ++u) fn(ctx, u);
    return;
  }
  if (nthreads > n) nthreads = n;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  unit_job* jobs = (unit_job*)malloc(sizeof(unit_job) * nthreads);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (unit_job){fn, ctx, n, nthreads, t};
    pthread_create(&th[t], NULL, unit_worker, &jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
}

/* ------------------------------------------------------------------------ */
/* Layer step over packed sequences: conv + split + norm + gates + rule      */
/* ------------------------------------------------------------------------ */
/*
 * A decode step is this with every sequence of length 1 and its initial state
 * taken from the slot.
 *
 * mixed_qkv  [Ttot, D] bf16 (pre-conv; already q|k|v when conv_w == NULL)
 * a, b       [Ttot, Hv] gate inputs (gate_direct selects their meaning)
 * conv_state pool of cache dtype / layout; ssm_state [num_slots, Hv, dv, dk]
 *            fp64 pool, in place
 * cu_seqlens [N+1], slot [N], has_init [N] (NULL = every sequence starts from
 *            the slot's state)
 * out        [Ttot, Hv, dv] fp64 (unrounded); out_bits [Ttot, Hv, dv] bf16 of
 *            the same (nullable)
 * head_mask  [Hv] (nullable): heads with mask 0 are skipped (their outputs and
 *            states untouched) -- lets large cases be sampled by head.
 * state_bf16 1: the pool holds bf16 values (exact in fp64); each call's final state
 *            is rounded to bf16 when stored, the arithmetic staying fp64.
 */
typedef struct {
  const uint16_t* y;   /* conv output bits [Ttot, D] */
  const void *a, *b;
  int gate_direct;
  const float *A_log, *dt_bias;
  double* ssm;
  const int32_t *cu, *slot;
  const uint8_t* has_init;
  int num_slots, Hk, Hv, dk, dv, D, qk_l2norm;
  double scale;
  double* out;
  uint16_t* out_bits;
  const uint8_t* head_mask;
  int state_bf16;  /* 1: the stored state is rounded to bf16 ([P1] Summary, state ABI) */
} rule_ctx;

static void rule_unit(void* p, int unit) {
  rule_ctx* c = (rule_ctx*)p;
  int i = unit / c->Hv, h = unit % c->Hv;
  if (c->head_mask && !c->head_mask[h]) return;
  int bos = c->cu[i], eos = c->cu[i + 1];
  int cls = slot_class(c->slot[i], c->num_slots);
  int dk = c->dk, dv = c->dv;
  if (cls <= 0) {
    for (int t = bos; t < eos; ++t)
      for (int r = 0; r < dv; ++r) {
        size_t o = ((size_t)t * c->Hv + h) * dv + r;
        c->out[o] = 0.0;
        if (c->out_bits) c->out_bits[o] = 0;
      }
    return;
  }
  int s = c->slot[i];
  int kh = h / (c->Hv / c->Hk);
  double* S = (double*)malloc(sizeof(double) * dv * dk);
  double* Sp = c->ssm + ((size_t)s * c->Hv + h) * dv * dk;
  if (c->has_init == NULL || c->has_init[i]) memcpy(S, Sp, sizeof(double) * dv * dk);
  else memset(S, 0, sizeof(double) * dv * dk);
  double* q = (double*)malloc(sizeof(double) * dk);
  double* k = (double*)malloc(sizeof(double) * dk);
  double* v = (double*)malloc(sizeof(double) * dv);
  double* o = (double*)malloc(sizeof(double) * dv);
  for (int t = bos; t < eos; ++t) {
    const uint16_t* y = c->y + (size_t)t * c->D;
    for (int j = 0; j < dk; ++j) {
      q[j] = bf16_to_f64(y[kh * dk + j]);
      k[j] = bf16_to_f64(y[c->Hk * dk + kh * dk + j]);
    }
    for (int r = 0; r < dv; ++r) v[r] = bf16_to_f64(y[2 * c->Hk * dk + h * dv + r]);
    qk_normalise(q, dk, c->qk_l2norm, c->scale);
    qk_normalise(k, dk, c->qk_l2norm, 1.0);
    double g, beta;
    gate_values(c->a, c->b, c->gate_direct, c->A_log, c->dt_bias, (size_t)t * c->Hv + h, h, &g,
                &beta);
    delta_rule_token(S, q, k, v, g, beta, dk, dv, o);
    for (int r = 0; r < dv; ++r) {
      size_t oi = ((size_t)t * c->Hv + h) * dv + r;
      c->out[oi] = o[r];
      if (c->out_bits) c->out_bits[oi] = gdn_ref_round_bf16(o[r]);
    }
  }
  /* bf16 storage: round once, at the write-back; the arithmetic stayed fp64 */
  if (c->state_bf16)
    for (int e = 0; e < dv * dk; ++e) S[e] = round_bf16_val(S[e]);
  memcpy(Sp, S, sizeof(double) * dv * dk);
  free(S); free(q); free(k); free(v); free(o);
}

typedef struct {
  const uint16_t* x;
  uint16_t* y;
  conv_pool pool;
  const uint16_t *w, *bias;
  int silu, D, W;
  const int32_t *cu, *slot;
  const uint8_t* has_init;
  int num_slots;
} conv_ctx;

static void conv_unit(void* p, int i) {
  conv_ctx* c = (conv_ctx*)p;
  int bos = c->cu[i], eos = c->cu[i + 1];
  int cls = slot_class(c->slot[i], c->num_slots);
  if (cls <= 0) {
    memset(c->y + (size_t)bos * c->D, 0, sizeof(uint16_t) * (size_t)(eos - bos) * c->D);
    return;
  }
  int s = c->slot[i], D = c->D, W = c->W;
  double* win = (double*)malloc(sizeof(double) * (size_t)D * (W - 1));
  int init = (c->has_init == NULL || c->has_init[i]);
  for (int ch = 0; ch < D; ++ch)
    for (int j = 0; j < W - 1; ++j)
      win[(size_t)ch * (W - 1) + j] = init ? conv_get(&c->pool, s, ch, j) : 0.0;
  for (int t = bos; t < eos; ++t)
    conv_row(win, c->x + (size_t)t * D, c->w, c->bias, D, W, c->pool.f32, c->silu,
             c->y + (size_t)t * D, NULL);
  for (int ch = 0; ch < D; ++ch)
    for (int j = 0; j < W - 1; ++j) conv_put(&c->pool, s, ch, j, win[(size_t)ch * (W - 1) + j]);
  free(win);
}

int gdn_ref_layer(const uint16_t* mixed_qkv, const void* a, const void* b, int gate_direct,
                  const float* A_log, const float* dt_bias, const uint16_t* conv_w,
                  const uint16_t* conv_b, int silu, void* conv_state, int conv_f32,
                  int conv_layout, double* ssm_state, const int32_t* cu_seqlens,
                  const int32_t* slot, const uint8_t* has_init, int N, int Ttot, int num_slots,
                  int Hk, int Hv, int dk, int dv, int W, double scale, int qk_l2norm,
                  double* out, uint16_t* out_bits, const uint8_t* head_mask, int nthreads,
                  int32_t* err, int state_bf16) {
  int D = 2 * Hk * dk + Hv * dv;
  if (Hk <= 0 || Hv % Hk != 0 || W < 2 || W > 16) return 1;
  for (int i = 0; i < N; ++i)
    if (slot_class(slot[i], num_slots) < 0 && err) *err |= 1;
  uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)Ttot * D + 1));
  if (conv_w) {
    conv_ctx cc = {mixed_qkv, y, {conv_state, conv_f32, conv_layout, D, W}, conv_w, conv_b,
                   silu, D, W, cu_seqlens, slot, has_init, num_slots};
    run_units(conv_unit, &cc, N, nthreads);
  } else {
    memcpy(y, mixed_qkv, sizeof(uint16_t) * (size_t)Ttot * D);
  }
  rule_ctx rc = {y, a, b, gate_direct, A_log, dt_bias, ssm_state, cu_seqlens, slot, has_init,
                 num_slots, Hk, Hv, dk, dv, D, qk_l2norm, scale, out, out_bits, head_mask,
                 state_bf16};
  run_units(rule_unit, &rc, N * Hv, nthreads);
  free(y);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Output gate: gated RMSNorm of o over each value head ([P1] page, Summary   */
/* by CodeRabbit: gated RMSNorm with SiLU or sigmoid gating; Walkthrough:     */
/* the weight offset)                                                         */
/* ------------------------------------------------------------------------ */

/* For each of `rows` vectors o[r][0..dv) (one token, one value head):
 *   y[i] = o[i] / sqrt(mean_j o[j]^2 + eps) * (w[i] + offset) * act(z[i]),
 * act = SiLU (z * sigmoid(z), act_kind 0) or sigmoid (act_kind 1). The norm is
 * taken before the gate (the GDN block normalises the core output, then gates
 * it with z). z arrives as bf16 bits, w as fp32; all arithmetic is fp64. The
 * pages leave 0/0 open: an all-zero head with eps = 0 gates to zero. */
void gdn_ref_gated_rmsnorm(const double* o, const uint16_t* z, const float* w, double offset,
                           double eps, int act_kind, int64_t rows, int dv, double* y) {
  for (int64_t r = 0; r < rows; ++r) {
    const double* orow = o + (size_t)r * dv;
    double ss = 0.0;
    for (int i = 0; i < dv; ++i) ss += orow[i] * orow[i];
    const double den = ss / dv + eps;
    const double inv = den > 0.0 ? 1.0 / sqrt(den) : 0.0; /* all-zero head, eps 0: zero out */
    for (int i = 0; i < dv; ++i) {
      const double zi = bf16_to_f64(z[(size_t)r * dv + i]);
      const double gate = act_kind == 0 ? zi * gdn_ref_sigmoid(zi) : gdn_ref_sigmoid(zi);
      y[(size_t)r * dv + i] = orow[i] * inv * ((double)w[i] + offset) * gate;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Planted mistake for the batch-invariance protocol (negative control)      */
/* ------------------------------------------------------------------------ */

/* Same as the head recurrence, but the predict dot product is summed in an
 * order that depends on the batch size B. Used only to show that the
 * batch-invariance test can fail. */
void gdn_ref_recurrent_head_batch_dependent(const double* q, const double* k, const double* v,
                                            const double* g, const double* beta, double* S,
                                            int T, int dk, int dv, int B, double* o) {
  for (int t = 0; t < T; ++t) {
    double alpha = exp(g[t]);
    const double* kt = k + (size_t)t * dk;
    const double* qt = q + (size_t)t * dk;
    for (int r = 0; r < dv; ++r) {
      double* Sr = S + (size_t)r * dk;
      for (int c = 0; c < dk; ++c) Sr[c] *= alpha;
      double pred = 0.0;
      if (B % 2) for (int c = dk - 1; c >= 0; --c) pred += Sr[c] * kt[c];
      else for (int c = 0; c < dk; ++c) pred += Sr[c] * kt[c];
      double delta = beta[t] * (v[(size_t)t * dv + r] - pred);
      for (int c = 0; c < dk; ++c) Sr[c] += delta * kt[c];
      double out = 0.0;
      for (int c = 0; c < dk; ++c) out += Sr[c] * qt[c];
      o[(size_t)t * dv + r] = out;
    }
  }
}
