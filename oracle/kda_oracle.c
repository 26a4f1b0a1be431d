/*
 * kda_oracle.c -- CPU oracle for the Kimi Delta Attention (KDA) layer core.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, token-by-token fp64
 * recurrence that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code, header, table or helper with the CUDA library, and the product path
 * never calls it.
 *
 * What it computes, per sequence, per head, per token t (the pages' order):
 *
 *   0. (optional) each of q, k, v passes through a causal depthwise
 *      convolution of width 4 over the tokens of its sequence, then Swish,
 *      x * sigmoid(x) ("Kimi K3's hybrid block, from first principles",
 *      section "From linear attention to the delta rule": queries and keys go
 *      through a short convolution of width 4, Swish and L2 normalisation,
 *      values through the convolution and Swish).  Taps w[c][0..3] weigh the
 *      raw rows t-3 .. t, oldest first; rows before the sequence start are
 *      the caller's window of earlier rows, zeros by default.  The
 *      convolution is the layer before the recurrence: its output is held in
 *      the data type of q, k, v (rounded to nearest-even bf16 for bf16 data,
 *      fp32 for fp32 data), as it would be when handed over by a separate
 *      convolution layer; from there on the arithmetic is fp64.  Storing is a
 *      quantisation, so for bf16 and fp32 data the value being stored is
 *      computed in the precision of the CUDA kernels: fp32, one fixed order of
 *      operations, and an exponential made of IEEE operations only (see
 *      conv_swish_f32).  fp64 data keeps an fp64 convolution and no rounding.
 *   1. q <- q / sqrt(sum q^2 + eps), k likewise (optional; the layer applies
 *      L2 normalisation to queries and keys: "Kimi K3's hybrid block, from
 *      first principles", section "From linear attention to the delta rule").
 *   2. beta <- sigmoid(beta) when beta is given as a logit (same section:
 *      beta_t is a sigmoid of a projection of the token).
 *   3. a = exp(clamp(log alpha, g_min, 0)), g_min = -5: the retention factor of
 *      every key channel lies in [e^-5, 1] ("Kimi K3", section "Forgetting
 *      different features at different rates"; the hybrid-block page, same
 *      section as above, on the bounded log-decay).  Optionally log alpha is
 *      formed from the decay logit z (a low-rank projection plus a per-channel
 *      bias b) with one scale A_h per head, through a bounded sigmoid:
 *      log alpha = g_min * sigmoid(A_h (z + b)) (same section: the log-decay is
 *      bounded from below with a learned per-head scale; "What changed": the
 *      mapping went from an unbounded softplus to a bounded sigmoid; the
 *      printed formula itself did not survive, this is the plainest form that
 *      keeps every factor in [e^g_min, 1]).
 *   4. S <- Diag(a) S                 (fade first)
 *   5. u = S^T k                      (what the memory now predicts for k)
 *   6. S <- S + beta k (v - u)^T      (erase the old association, write v)
 *      Steps 4-6 equal S_t = (I - beta k k^T) Diag(a) S_{t-1} + beta k v^T.
 *      The order fade -> erase -> write is the one stated on "Kimi K3,
 *      explained", section "Kimi Delta Attention: making the radical option
 *      work" (change one: erase, then write); the per-channel decay is that
 *      page's change two and the hybrid-block page's KDA definition.
 *   7. o_t = q_scale * S^T q          (q reads the UPDATED state: same page,
 *                                      the one-token-step figure)
 *
 * The optional epilogue (kda_oracle_gated_rmsnorm) is the per-head RMSNorm
 * times a full-rank sigmoid gate of the token ("Kimi K3's hybrid block",
 * section "From linear attention to the delta rule", last paragraph).
 *
 * Readings of what the pages leave open (eps values, clamp to 0 from above,
 * q_scale = 1) are fixed by the caller through kda_oracle_opts.
 *
 * Element types of the inputs: 0 = fp32, 1 = bf16 (raw 16-bit patterns),
 * 2 = fp64.  Every input element is widened exactly to double before use, so
 * that only the arithmetic of the implementation under test is measured.
 *
 * Compile-time switch KDA_ORACLE_MUTATION (tests only): plants one known
 * mistake so that the test suite can show its pins catch it.  Unset (0) in
 * every normal build.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef KDA_ORACLE_MUTATION
#define KDA_ORACLE_MUTATION 0
#endif

typedef struct {
  int l2norm_qk;     /* 1: L2-normalise q and k per head per token            */
  int beta_is_logit; /* 1: beta input is a logit, apply sigmoid               */
  double g_min;      /* floor of log alpha (the pages' value is -5)          */
  double q_scale;    /* multiplier on the read-out (1 by default)            */
  double eps_l2;     /* epsilon inside the L2-norm square root                */
  int decay_from_logit;      /* 1: log_alpha holds decay logits z; log alpha =
                                g_min * sigmoid(A_h (z + b_{h,c}))            */
  const double* decay_scale; /* A [H], NULL = ones                            */
  const double* decay_bias;  /* b [H][dk], NULL = zeros                       */
  const double* conv_weight; /* NULL: no short convolution.  Else taps
                                [3 (q, k, v)][H][d][4], oldest row first
                                (needs dk == dv == d)                        */
} kda_oracle_opts;

/* Raw rows of q, k, v before the current token, per tensor the 3 previous
 * rows oldest first: hist[(X * 3 + j) * d + c]. */
enum { CONV_W = 4, CONV_HIST = CONV_W - 1 };

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* Widen element i of a typed buffer to double (exact for all three types). */
static double load_elem(const void* p, int dtype, size_t i) {
  if (dtype == ORC_F64) return ((const double*)p)[i];
#if KDA_ORACLE_MUTATION == 11
  if (dtype == ORC_F32) { /* planted mistake: fp32 cut to its upper 16 bits */
    float f32 = ((const float*)p)[i];
    uint32_t b32;
    memcpy(&b32, &f32, sizeof b32);
    b32 &= 0xFFFF0000u;
    memcpy(&f32, &b32, sizeof f32);
    return (double)f32;
  }
#else
  if (dtype == ORC_F32) return (double)((const float*)p)[i];
#endif
  /* bf16: the upper 16 bits of an IEEE binary32 pattern */
#if KDA_ORACLE_MUTATION == 10
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 15; /* planted: wrong shift */
#else
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
#endif
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int dtype_ok(int d) { return d == ORC_F32 || d == ORC_BF16 || d == ORC_F64; }

/* Step 1 of the list above: x <- x / sqrt(sum x^2 + eps). */
static void l2_normalise(double* x, int n, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) x[i] *= inv;
}

/*
 * One token of the recurrence, steps 3-7.  S is [dk][dv] row-major, q and k
 * already normalised (if asked), beta already activated.  Writes o[dv].
 */
static void token_step(double* S, int dk, int dv, const double* q,
                       const double* k, const double* v, const double* log_a,
                       double beta, const kda_oracle_opts* opt, double* u,
                       double* o) {
  /* 3-4: fade each key channel (row c of S) by its own retention factor. */
#if KDA_ORACLE_MUTATION != 1 && KDA_ORACLE_MUTATION != 7
  for (int c = 0; c < dk; ++c) {
    double la = log_a[c];
#if KDA_ORACLE_MUTATION != 6
    if (la < opt->g_min) la = opt->g_min;
    if (la > 0.0) la = 0.0;
#endif
    double a = exp(la);
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
  }
#endif

#if KDA_ORACLE_MUTATION == 2
  /* planted mistake: read the state before the write */
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * q[c];
    o[j] = opt->q_scale * acc;
  }
#endif

  /* 5: u = S^T k */
  for (int j = 0; j < dv; ++j) u[j] = 0.0;
  for (int c = 0; c < dk; ++c) {
#if KDA_ORACLE_MUTATION == 9
    const double kc = q[c]; /* planted mistake: probe with the query */
#else
    const double kc = k[c];
#endif
    for (int j = 0; j < dv; ++j) u[j] += S[(size_t)c * dv + j] * kc;
  }

  /* 6: S <- S + beta k (v - u)^T */
  for (int c = 0; c < dk; ++c) {
#if KDA_ORACLE_MUTATION == 5
    const double bk = k[c]; /* planted mistake: beta dropped */
#else
    const double bk = beta * k[c];
#endif
    for (int j = 0; j < dv; ++j) {
#if KDA_ORACLE_MUTATION == 3
      S[(size_t)c * dv + j] += bk * (v[j] + u[j]); /* planted: wrong sign */
#else
      S[(size_t)c * dv + j] += bk * (v[j] - u[j]);
#endif
    }
  }

#if KDA_ORACLE_MUTATION == 7
  /* planted mistake: fade after the write (and erase on the unfaded state) */
  for (int c = 0; c < dk; ++c) {
    double la = log_a[c];
    if (la < opt->g_min) la = opt->g_min;
    if (la > 0.0) la = 0.0;
    double a = exp(la);
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
  }
#endif

  /* 7: o = q_scale * S^T q, from the updated state */
#if KDA_ORACLE_MUTATION != 2
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) {
#if KDA_ORACLE_MUTATION == 4
      acc += S[(size_t)(dk - 1 - c) * dv + j] * q[c]; /* planted: wrong row */
#else
      acc += S[(size_t)c * dv + j] * q[c];
#endif
    }
    o[j] = opt->q_scale * acc;
  }
#endif
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* x held in storage type `dtype`: fp32 by the C conversion (round to nearest),
 * bf16 by rounding that binary32 pattern to its upper 16 bits, to nearest
 * with ties to even; fp64 unchanged. */
static double store_as(double x, int dtype) {
  if (dtype == ORC_F64) return x;
  float f = (float)x;
  if (dtype == ORC_BF16) {
    uint32_t b;
    memcpy(&b, &f, sizeof b);
#if KDA_ORACLE_MUTATION != 18
    b += 0x7FFFu + ((b >> 16) & 1u);
#endif
    b &= 0xFFFF0000u; /* (mutation 18 plants truncation instead of rounding) */
    memcpy(&f, &b, sizeof f);
  }
  return (double)f;
}

/* e^t for fp32 t in [-80, 80] from IEEE operations only, so that any
 * implementation of the same steps gets the same bits: Cody and Waite's range
 * reduction t = n ln2 + r (n = rint(t log2 e), ln2 split into a 14-bit head,
 * exact in n * head, and a tail), then the Taylor polynomial of e^r to degree
 * 6 (|r| <= 0.35) by Horner's rule, scaled by 2^n. */
static float exp_f32(float t) {
  const float n = rintf(t * 0x1.715476p+0f);
  float r = fmaf(-n, 0x1.62e4p-1f, t);
  r = fmaf(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.6c16c2p-10f;     /* 1/720 */
  p = fmaf(p, r, 0x1.111112p-7f); /* 1/120 */
  p = fmaf(p, r, 0x1.555556p-5f); /* 1/24  */
  p = fmaf(p, r, 0x1.555556p-3f); /* 1/6   */
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return ldexpf(p, (int)n);
}

/* The stored value of the convolution + Swish in fp32 (the kernels'
 * precision): y = w3 x3 + w2 x2 + w1 x1 + w0 x0 accumulated in that order by
 * fused multiply-adds (x0 the oldest row), then y * sigmoid(y) with
 * sigmoid(y) = 1 / (1 + e^-y), the exponent clamped to [-80, 80]. */
static float conv_swish_f32(const double* wc, const double* xs) {
  const float w0 = (float)wc[0], w1 = (float)wc[1], w2 = (float)wc[2], w3 = (float)wc[3];
  float y = w3 * (float)xs[3];
  y = fmaf(w2, (float)xs[2], y);
  y = fmaf(w1, (float)xs[1], y);
  y = fmaf(w0, (float)xs[0], y);
  float t = -y;
  t = t < -80.0f ? -80.0f : (t > 80.0f ? 80.0f : t);
  const float sg = 1.0f / (1.0f + exp_f32(t));
  return y * sg;
}

/* Step 0 for one tensor X (0 = q, 1 = k, 2 = v) of one (token, head h of H):
 * x holds the raw row and receives conv + Swish; the raw row enters the
 * history. */
static void conv_swish(double* x, int X, int H, int h, int d, int dtype,
                       const kda_oracle_opts* opt, double* hist) {
  double* hx = hist + (size_t)X * CONV_HIST * d;
  for (int c = 0; c < d; ++c) {
    const double* wc0 = opt->conv_weight + (((size_t)X * H + h) * d + c) * CONV_W;
    /* the taps in the order they weigh the rows: oldest row first */
    double wc[CONV_W];
    for (int j = 0; j < CONV_W; ++j) {
#if KDA_ORACLE_MUTATION == 12
      wc[j] = wc0[CONV_W - 1 - j]; /* planted mistake: taps applied newest row first */
#else
      wc[j] = wc0[j];
#endif
    }
    const double xs[CONV_W] = {hx[c], hx[(size_t)d + c], hx[(size_t)2 * d + c], x[c]};
    for (int j = 0; j + 1 < CONV_HIST; ++j) hx[(size_t)j * d + c] = hx[(size_t)(j + 1) * d + c];
    hx[(size_t)(CONV_HIST - 1) * d + c] = x[c];
#if KDA_ORACLE_MUTATION == 13
    const int swish = X != 2; /* planted mistake: no Swish on v */
#else
    const int swish = 1;
#endif
    if (dtype == ORC_F64) {
      double y = 0.0;
      for (int j = 0; j < CONV_W; ++j) y += wc[j] * xs[j];
      x[c] = swish ? y * sigmoid(y) : y;
    } else if (swish) {
      x[c] = store_as((double)conv_swish_f32(wc, xs), dtype);
    } else {
      x[c] = store_as(wc[3] * xs[3] + wc[2] * xs[2] + wc[1] * xs[1] + wc[0] * xs[0], dtype);
    }
  }
}

/* Steps 0-3 for one (token, head): widen, convolve (optional), normalise and
 * activate.  hist: the raw-row history of this (sequence, head), used and
 * advanced when the convolution is on. */
static void prologue(const void* q, const void* k, const void* v, int qkv_dtype,
                     const void* log_alpha, int la_dtype, const void* beta,
                     int beta_dtype, size_t row, int H, int h, int dk, int dv,
                     const kda_oracle_opts* opt, double* hist, double* qd,
                     double* kd, double* vd, double* lad, double* bd) {
  const size_t qk_off = (row * (size_t)H + (size_t)h) * (size_t)dk;
  const size_t v_off = (row * (size_t)H + (size_t)h) * (size_t)dv;
  for (int c = 0; c < dk; ++c) {
    qd[c] = load_elem(q, qkv_dtype, qk_off + c);
    kd[c] = load_elem(k, qkv_dtype, qk_off + c);
    lad[c] = load_elem(log_alpha, la_dtype, qk_off + c);
  }
  for (int j = 0; j < dv; ++j) vd[j] = load_elem(v, qkv_dtype, v_off + j);
  if (opt->conv_weight) {
    conv_swish(qd, 0, H, h, dk, qkv_dtype, opt, hist);
    conv_swish(kd, 1, H, h, dk, qkv_dtype, opt, hist);
    conv_swish(vd, 2, H, h, dv, qkv_dtype, opt, hist);
  }
  if (opt->decay_from_logit) {
    const double A = opt->decay_scale ? opt->decay_scale[h] : 1.0;
    for (int c = 0; c < dk; ++c) {
      const double z = lad[c] + (opt->decay_bias ? opt->decay_bias[(size_t)h * dk + c] : 0.0);
#if KDA_ORACLE_MUTATION == 14
      lad[c] = -log1p(exp(A * z)); /* planted mistake: the old unbounded softplus */
#elif KDA_ORACLE_MUTATION == 15
      lad[c] = A * opt->g_min * sigmoid(z); /* planted mistake: scale outside */
#else
      lad[c] = opt->g_min * sigmoid(A * z);
#endif
    }
  }
  double b = load_elem(beta, beta_dtype, row * (size_t)H + (size_t)h);
  if (opt->beta_is_logit) b = sigmoid(b);
  *bd = b;
  if (opt->l2norm_qk) {
    l2_normalise(qd, dk, opt->eps_l2);
#if KDA_ORACLE_MUTATION != 8
    l2_normalise(kd, dk, opt->eps_l2);
#endif
  }
}

/* History of one (sequence n, head h) from the caller's window
 * conv_state [N][3][3][H][d] (fp64, NULL = zeros). */
static void init_hist(double* hist, const double* conv_state, int n, int H, int h, int d) {
  for (int X = 0; X < 3; ++X)
    for (int j = 0; j < CONV_HIST; ++j)
      for (int c = 0; c < d; ++c) {
#if KDA_ORACLE_MUTATION == 16
        const int jj = CONV_HIST - 1 - j; /* planted mistake: window read newest first */
#else
        const int jj = j;
#endif
        hist[((size_t)X * CONV_HIST + j) * d + c] =
            conv_state ? conv_state[((((size_t)n * 3 + X) * CONV_HIST + jj) * H + h) * d + c]
                       : 0.0;
      }
}

/* Back into the caller's window. */
static void store_hist(const double* hist, double* conv_state, int n, int H, int h, int d) {
  for (int X = 0; X < 3; ++X)
    for (int j = 0; j < CONV_HIST; ++j)
      for (int c = 0; c < d; ++c)
        conv_state[((((size_t)n * 3 + X) * CONV_HIST + j) * H + h) * d + c] =
            hist[((size_t)X * CONV_HIST + j) * d + c];
}

/*
 * Prefill over a packed batch of N sequences (cu_seqlens[N+1] on the host,
 * NULL = N equal-length sequences of T_total/N tokens).
 *
 *   q, k        [T_total][H][dk]  (qkv_dtype)
 *   v           [T_total][H][dv]  (qkv_dtype)
 *   log_alpha   [T_total][H][dk]  (la_dtype)
 *   beta        [T_total][H]      (beta_dtype)
 *   S0          [N][H][dk][dv] fp64, NULL = zeros
 *   heads h0 .. h0+nh-1 are computed (a subset keeps full-size checks cheap)
 *   o           [T_total][nh][dv] fp64 out
 *   S_T         [N][nh][dk][dv]   fp64 out (NULL = not wanted)
 *   conv_state  [N][3][3][H][d] fp64, NULL = zeros: with opt->conv_weight, the
 *               raw q, k, v rows of the 3 tokens before each sequence, oldest
 *               first (read only)
 *
 * Returns 0, or -1 on a bad argument.
 */
int kda_oracle_prefill(const void* q, const void* k, const void* v, int qkv_dtype,
                       const void* log_alpha, int la_dtype, const void* beta,
                       int beta_dtype, const double* S0,
                       const int32_t* cu_seqlens, int N, int T_total, int H,
                       int dk, int dv, int h0, int nh,
                       const kda_oracle_opts* opt, double* o, double* S_T,
                       const double* conv_state) {
  if (!q || !k || !v || !log_alpha || !beta || !o || !opt) return -1;
  if (N < 1 || T_total < 0 || H < 1 || dk < 1 || dv < 1) return -1;
  if (opt->conv_weight && dk != dv) return -1;
  if (h0 < 0 || nh < 1 || h0 + nh > H) return -1;
  if (!dtype_ok(qkv_dtype) || !dtype_ok(la_dtype) || !dtype_ok(beta_dtype)) return -1;
  if (!cu_seqlens && (T_total % N) != 0) return -1;
  if (cu_seqlens) {
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return -1;
    for (int n = 0; n < N; ++n)
      if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  }
  const int units = N * nh;
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int unit = 0; unit < units; ++unit) {
    const int n = unit / nh, hh = unit % nh, h = h0 + hh;
    const int t0 = cu_seqlens ? cu_seqlens[n] : n * (T_total / N);
    const int t1 = cu_seqlens ? cu_seqlens[n + 1] : (n + 1) * (T_total / N);
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(3 * dk + 3 * dv + 9 * dk));
    if (!S || !buf) {
      free(S);
      free(buf);
#pragma omp atomic write
      failed = 1;
      continue;
    }
    double *qd = buf, *kd = buf + dk, *lad = buf + 2 * dk;
    double *vd = buf + 3 * dk, *u = vd + dv, *ot = u + dv, *hist = ot + dv;
    const size_t SS = (size_t)dk * dv;
    if (S0) memcpy(S, S0 + ((size_t)n * H + h) * SS, sizeof(double) * SS);
    else memset(S, 0, sizeof(double) * SS);
    if (opt->conv_weight) init_hist(hist, conv_state, n, H, h, dk);
#if KDA_ORACLE_MUTATION == 17
    /* planted mistake: the window is the packed rows before the sequence,
       whichever sequence they belong to */
    if (opt->conv_weight && t0 >= CONV_HIST)
      for (int j = 0; j < CONV_HIST; ++j)
        for (int c = 0; c < dk; ++c) {
          const size_t off = ((size_t)(t0 - CONV_HIST + j) * H + h) * dk + c;
          hist[(0 * CONV_HIST + j) * (size_t)dk + c] = load_elem(q, qkv_dtype, off);
          hist[(1 * CONV_HIST + j) * (size_t)dk + c] = load_elem(k, qkv_dtype, off);
          hist[(2 * CONV_HIST + j) * (size_t)dk + c] = load_elem(v, qkv_dtype, off);
        }
#endif
    for (int t = t0; t < t1; ++t) {
      double b;
      prologue(q, k, v, qkv_dtype, log_alpha, la_dtype, beta, beta_dtype,
               (size_t)t, H, h, dk, dv, opt, hist, qd, kd, vd, lad, &b);
      token_step(S, dk, dv, qd, kd, vd, lad, b, opt, u, ot);
      memcpy(o + ((size_t)t * nh + hh) * dv, ot, sizeof(double) * dv);
    }
    if (S_T) memcpy(S_T + ((size_t)n * nh + hh) * SS, S, sizeof(double) * SS);
    free(S);
    free(buf);
  }
  return failed ? -1 : 0;
}

/*
 * One recurrent decode step for N independent sequences, state updated in
 * place: the same token recurrence as above, applied once.
 *   q, k [N][H][dk]; v [N][H][dv]; log_alpha [N][H][dk]; beta [N][H];
 *   S [N][H][dk][dv] fp64 in/out; o [N][H][dv] fp64 out;
 *   conv_state [N][3][3][H][d] fp64 in/out with opt->conv_weight (the raw
 *   rows of the 3 previous tokens, oldest first; NULL = zeros, not kept).
 */
int kda_oracle_decode_step(const void* q, const void* k, const void* v,
                           int qkv_dtype, const void* log_alpha, int la_dtype,
                           const void* beta, int beta_dtype, double* S, int N,
                           int H, int dk, int dv, const kda_oracle_opts* opt,
                           double* o, double* conv_state) {
  if (!q || !k || !v || !log_alpha || !beta || !S || !o || !opt) return -1;
  if (N < 1 || H < 1 || dk < 1 || dv < 1) return -1;
  if (opt->conv_weight && dk != dv) return -1;
  if (!dtype_ok(qkv_dtype) || !dtype_ok(la_dtype) || !dtype_ok(beta_dtype)) return -1;
  const int units = N * H;
  int failed = 0;
#pragma omp parallel for schedule(static)
  for (int unit = 0; unit < units; ++unit) {
    const int n = unit / H, h = unit % H;
    double* buf = (double*)malloc(sizeof(double) * (size_t)(3 * dk + 3 * dv + 9 * dk));
    if (!buf) {
#pragma omp atomic write
      failed = 1;
      continue;
    }
    double *qd = buf, *kd = buf + dk, *lad = buf + 2 * dk;
    double *vd = buf + 3 * dk, *u = vd + dv, *ot = u + dv, *hist = ot + dv;
    double b;
    if (opt->conv_weight) init_hist(hist, conv_state, n, H, h, dk);
    prologue(q, k, v, qkv_dtype, log_alpha, la_dtype, beta, beta_dtype,
             (size_t)n, H, h, dk, dv, opt, hist, qd, kd, vd, lad, &b);
    if (opt->conv_weight && conv_state) store_hist(hist, conv_state, n, H, h, dk);
    token_step(S + (size_t)unit * dk * dv, dk, dv, qd, kd, vd, lad, b, opt, u, ot);
    memcpy(o + (size_t)unit * dv, ot, sizeof(double) * dv);
    free(buf);
  }
  return failed ? -1 : 0;
}

/*
 * Per-head RMSNorm times a sigmoid gate:
 *   y[r][h][j] = o[r][h][j] / sqrt(mean_j o[r][h][:]^2 + eps) * w[j] * sigmoid(gate[r][h0+h][j])
 *   o, y  [rows][nh][dv] fp64;  gate [rows][H][dv] (gate_dtype), heads h0..h0+nh-1;
 *   w     [dv] fp64 or NULL (= ones).
 */
int kda_oracle_gated_rmsnorm(const double* o, int rows, int nh, int dv,
                             const void* gate, int gate_dtype, int H, int h0,
                             const double* w, double eps, double* y) {
  if (!o || !gate || !y || rows < 0 || nh < 1 || dv < 1 || H < 1) return -1;
  if (h0 < 0 || h0 + nh > H || !dtype_ok(gate_dtype)) return -1;
  const long units = (long)rows * nh;
#pragma omp parallel for schedule(static)
  for (long unit = 0; unit < units; ++unit) {
    const long r = unit / nh;
    const int hh = (int)(unit % nh);
    const double* x = o + (size_t)unit * dv;
    double ss = 0.0;
    for (int j = 0; j < dv; ++j) ss += x[j] * x[j];
    const double inv = 1.0 / sqrt(ss / dv + eps);
    for (int j = 0; j < dv; ++j) {
      double g = load_elem(gate, gate_dtype, ((size_t)r * H + h0 + hh) * dv + j);
      double sg = 1.0 / (1.0 + exp(-g));
      double wj = w ? w[j] : 1.0;
      y[(size_t)unit * dv + j] = x[j] * inv * wj * sg;
    }
  }
  return 0;
}

/* Mutation number this build was compiled with (0 = faithful build). */
int kda_oracle_mutation(void) { return KDA_ORACLE_MUTATION; }
