/*
 * gdn_oracle.c -- plain, slow, token-by-token fp64 CPU oracle for the gated
 * delta rule forward, its backward (the exact gradient of that forward) and
 * the steps around it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file: it is used by tests/, by __graft_entry__.smoke() and by
 * the cpu_baseline / reference leg of bench.py.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources for what is computed (cited by page title and section):
 *  - "feat: hybrid CP for Qwen3.5 MoE (DeltaNet + attention)", Summary: the
 *    DeltaNet layer keeps a recurrent state matrix per head that is updated
 *    token after token; Approach / communication-cost table: only that state
 *    (H x K x (K+V) numbers) has to cross a sequence split.
 *  - The gated delta rule itself (Yang, Kautz, Hatamizadeh, "Gated Delta
 *    Networks: Improving Mamba2 with Delta Rule", ICLR 2025), in the form
 *        S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *        o_t = scale * S_t q_t,          S_t in R^{V x K}, fp32 on the GPU.
 *  - "[v1] support GDN Ulysses cp", What This PR Does / Key decisions 2, 4-6:
 *    the layer's parameters A_log and dt_bias, inputs a and b, the causal
 *    conv1d over concatenated Q|K|V channels with cu_seqlens so packed samples
 *    never mix, and cu_seqlens derived from position_ids.
 *  - "Qwen3.5 cp - #1", Architecture: a sequence split into segments, each
 *    summarised by a local state b and a transition M, then an fp32 chain
 *    reduce of the (b, M) pairs across segments.
 *
 * Every routine below is the definition written out as loops in double
 * precision, with no blocking, fusion or reordering beyond what the
 * definition states.  Layouts are token-major and contiguous:
 *   q, k   [n_tok, Hqk, K]      v, o  [n_tok, Hv, V]
 *   g, beta[n_tok, Hv]          h0, hT, S_local, S_start [n_seq, Hv, V, K]
 *   M      [n_seg, Hv, K, K]    x, y  [n_tok, C]   w [C, W]
 * A sequence s covers tokens [cu[s], cu[s+1]) of the flattened token axis.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ gates */

/* Qwen3.5 GatedDeltaNet gates ("[v1] support GDN Ulysses cp", What This PR
 * Does: A_log and dt_bias are per-v-head layer parameters, a and b are
 * per-token projections):
 *    g    = -exp(A_log[h]) * softplus(a + dt_bias[h])   (log of the decay)
 *    beta = sigmoid(b)                                    (write strength)
 * softplus(x) = log(1 + e^x), evaluated as max(x,0) + log1p(exp(-|x|)) so
 * that it neither overflows nor loses the small-x digits. */
void oracle_gate_prep(const double *a, const double *b, const double *A_log,
                      const double *dt_bias, int64_t n_tok, int Hv, double *g,
                      double *beta) {
  for (int64_t t = 0; t < n_tok; ++t) {
    for (int h = 0; h < Hv; ++h) {
      const int64_t i = t * Hv + h;
      const double x = a[i] + dt_bias[h];
      const double softplus = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
      g[i] = -exp(A_log[h]) * softplus;
      beta[i] = 1.0 / (1.0 + exp(-b[i]));
    }
  }
}

/* ------------------------------------------------------------------- conv */

/* Depthwise causal conv1d over channels, one sequence at a time
 * ("[v1] support GDN Ulysses cp", Key decisions 5: causal_conv1d_fn is given
 * cu_seqlens so no sample reads another sample's tokens).  Cross-correlation
 * order, as in torch's conv1d with left padding W-1: tap W-1 multiplies the
 * current token, tap 0 the token W-1 steps back.  Tokens before the start of
 * the sequence read as zero.  act = 1 applies SiLU, x * sigmoid(x). */
void oracle_conv1d(const double *x, const double *w, const double *bias,
                   const int32_t *cu, int n_seq, int C, int W, int act,
                   double *y) {
  for (int s = 0; s < n_seq; ++s) {
    for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
      for (int c = 0; c < C; ++c) {
        double acc = bias ? bias[c] : 0.0;
        for (int j = 0; j < W; ++j) {
          const int64_t src = t - (W - 1) + j;
          if (src >= cu[s]) acc += w[(int64_t)c * W + j] * x[src * C + c];
        }
        y[t * C + c] = act ? acc / (1.0 + exp(-acc)) : acc;
      }
    }
  }
}

/* x / sqrt(sum x^2 + eps): unit-norm queries and keys; eps keeps a zero
 * vector at zero. */
static void l2_normalise(const double *x, int n, double eps, double *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv;
}

void oracle_l2norm_rows(const double *x, int64_t rows, int n, double eps,
                        double *out) {
  for (int64_t r = 0; r < rows; ++r) l2_normalise(x + r * n, n, eps, out + r * n);
}

/* Gated RMS norm of the core's output ("[v1] support GDN Ulysses cp", Design: the layer
 * applies a norm to the chunk_gated_delta_rule output, and z is one of the layer's
 * per-token components).  The pages give no formula; the reading taken is the gated
 * RMS norm over each (token, v-head) row of V values:
 *    y[v] = o[v] / sqrt(mean_v o^2 + eps) * w[v] * z[v] * sigmoid(z[v])
 * with w [V] (NULL reads as ones). */
void oracle_gated_rmsnorm(const double *o, const double *z, const double *w, int64_t rows,
                          int V, double eps, double *y) {
  for (int64_t r = 0; r < rows; ++r) {
    const double *orow = o + r * V, *zrow = z + r * V;
    double ms = 0.0;
    for (int v = 0; v < V; ++v) ms += orow[v] * orow[v];
    ms /= (double)V;
    const double inv = 1.0 / sqrt(ms + eps);
    for (int v = 0; v < V; ++v) {
      const double gate = zrow[v] / (1.0 + exp(-zrow[v]));
      y[r * V + v] = orow[v] * inv * (w ? w[v] : 1.0) * gate;
    }
  }
}

/* ------------------------------------------------------ thread work queue */

typedef struct {
  void (*fn)(void *ctx, int64_t job);
  void *ctx;
  int64_t n_jobs;
  int64_t next; /* shared counter, taken with an atomic add */
} queue_t;

static void *queue_worker(void *arg) {
  queue_t *q = (queue_t *)arg;
  for (;;) {
    const int64_t j = __atomic_fetch_add(&q->next, 1, __ATOMIC_RELAXED);
    if (j >= q->n_jobs) break;
    q->fn(q->ctx, j);
  }
  return NULL;
}

/* Runs fn(ctx, j) for j in [0, n_jobs) on n_threads threads.  Jobs write
 * disjoint outputs, so the result does not depend on the thread count. */
static void run_jobs(void (*fn)(void *, int64_t), void *ctx, int64_t n_jobs,
                     int n_threads) {
  queue_t q = {fn, ctx, n_jobs, 0};
  if (n_threads <= 1 || n_jobs <= 1) {
    queue_worker(&q);
    return;
  }
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 0; i < n_threads; ++i)
    if (pthread_create(&th[i], NULL, queue_worker, &q) == 0) ++started;
  if (started == 0) queue_worker(&q);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------ the recurrence */

typedef struct {
  const double *q, *k, *v, *g, *beta, *h0;
  const int32_t *cu;
  int n_seq, Hqk, Hv, K, V, l2norm;
  double scale, eps;
  double *o, *hT;
} fwd_ctx;

/* One token's state update, S_t from S_{t-1}: S <- alpha S;  r = v - S k;
 * S <- S + beta r k^T. */
static void fwd_token(double *S, const double *kt, const double *vt, double alpha, double bt,
                      int K, int V) {
  for (int i = 0; i < V; ++i) {
    double *row = S + (int64_t)i * K;
    double pred = 0.0;
    for (int j = 0; j < K; ++j) {
      row[j] *= alpha;
      pred += row[j] * kt[j];
    }
    const double r = vt[i] - pred;
    for (int j = 0; j < K; ++j) row[j] += bt * r * kt[j];
  }
}

/* One (sequence, v-head) pair, token by token.  The v-head h reads q/k head
 * h / (Hv / Hqk): each q/k head serves Hv/Hqk consecutive v-heads.
 * Per token, with alpha = exp(g_t):
 *     S <- alpha * S                      (decay)
 *     r  = v_t - S k_t                    (what the state predicts wrongly)
 *     S <- S + beta_t * r k_t^T           (delta-rule write)
 *     o_t = scale * S q_t
 * which expands to S_t = alpha S_{t-1} (I - beta k k^T) + beta v k^T. */
static void fwd_job(void *vctx, int64_t job) {
  const fwd_ctx *c = (const fwd_ctx *)vctx;
  const int s = (int)(job / c->Hv), h = (int)(job % c->Hv);
  const int K = c->K, V = c->V, qh = h / (c->Hv / c->Hqk);
  double *S = (double *)calloc((size_t)V * K, sizeof(double));
  double *kt = (double *)malloc(sizeof(double) * K);
  double *qt = (double *)malloc(sizeof(double) * K);
  if (c->h0) memcpy(S, c->h0 + ((int64_t)s * c->Hv + h) * V * K, sizeof(double) * V * K);
  for (int64_t t = c->cu[s]; t < c->cu[s + 1]; ++t) {
    const double *kraw = c->k + (t * c->Hqk + qh) * K;
    const double *qraw = c->q + (t * c->Hqk + qh) * K;
    if (c->l2norm) {
      l2_normalise(kraw, K, c->eps, kt);
      l2_normalise(qraw, K, c->eps, qt);
    } else {
      memcpy(kt, kraw, sizeof(double) * K);
      memcpy(qt, qraw, sizeof(double) * K);
    }
    const double alpha = exp(c->g[t * c->Hv + h]);
    const double bt = c->beta[t * c->Hv + h];
    const double *vt = c->v + (t * c->Hv + h) * V;
    double *ot = c->o + (t * c->Hv + h) * V;
    fwd_token(S, kt, vt, alpha, bt, K, V);
    for (int i = 0; i < V; ++i) {
      const double *row = S + (int64_t)i * K;
      double out = 0.0;
      for (int j = 0; j < K; ++j) out += row[j] * qt[j];
      ot[i] = c->scale * out;
    }
  }
  if (c->hT) memcpy(c->hT + ((int64_t)s * c->Hv + h) * V * K, S, sizeof(double) * V * K);
  free(S);
  free(kt);
  free(qt);
}

/* o and the final state hT of every sequence and v-head.  h0 may be NULL
 * (zero start state); hT may be NULL. */
void oracle_gdn_fwd(const double *q, const double *k, const double *v,
                    const double *g, const double *beta, const double *h0,
                    const int32_t *cu, int n_seq, int Hqk, int Hv, int K, int V,
                    double scale, int l2norm, double eps, double *o, double *hT,
                    int n_threads) {
  fwd_ctx c = {q, k, v, g, beta, h0, cu, n_seq, Hqk, Hv, K, V, l2norm, scale, eps, o, hT};
  run_jobs(fwd_job, &c, (int64_t)n_seq * Hv, n_threads);
}

/* ------------------------------------------------ the recurrence, backward */

/* The backward of the chunked rule is what training runs through the layer
 * ("[v1] support GDN Ulysses cp", Testing: loss alignment over 2000 training
 * steps; "feat: hybrid CP for Qwen3.5 MoE (DeltaNet + attention)", Test plan:
 * forward/backward passes).  The pages give no formula for it, so it is the
 * exact gradient of the forward above: for upstream gradients dout (of o) and
 * dhT (of hT), the gradients of
 *     L = sum_t <dout_t, o_t> + sum <dhT, S_T>
 * with respect to q, k, v, g, beta and h0, taken back through each token step
 * of fwd_job in reverse order.  With P = alpha S_{t-1}, r = v - P k,
 * S_t = P + beta r k^T and o_t = scale S_t q, given dS = dL/dS_t:
 *     dq   += scale S_t^T dout_t         dS  += scale dout_t q^T
 *     dbeta = r^T dS k                    dr   = beta dS k,   dv = dr
 *     dk   += beta dS^T r - P^T dr        dP   = dS - dr k^T
 *     dg    = alpha <S_{t-1}, dP>         dS_{t-1} = alpha dP
 * and dh0 = dS_0.  q and k here are the unit-norm vectors when l2norm is set;
 * their gradients then go back through the norm (l2_backward).  A q/k head
 * serves Hv/Hqk v-heads, so its gradient is the sum over them. */

typedef struct {
  const double *q, *k, *v, *g, *beta, *h0, *dout, *dhT;
  const int32_t *cu;
  int n_seq, Hqk, Hv, K, V, l2norm;
  double scale, eps;
  double *dq, *dk, *dv, *dg, *dbeta, *dh0;
} bwd_ctx;

enum { kCheckpoint = 64 }; /* tokens between the states kept from the forward */

/* With n = sqrt(|x|^2 + eps) and xh = x / n:  dx = dxh / n - x (x . dxh) / n^3. */
static void l2_backward(const double *x, const double *dxh, int n, double eps, double *dx) {
  double ss = 0.0, xd = 0.0;
  for (int i = 0; i < n; ++i) {
    ss += x[i] * x[i];
    xd += x[i] * dxh[i];
  }
  const double nn = sqrt(ss + eps);
  for (int i = 0; i < n; ++i) dx[i] = dxh[i] / nn - x[i] * xd / (nn * nn * nn);
}

/* One (sequence, q/k head) pair: its Hv/Hqk v-heads one after another.  The
 * forward keeps the state before every kCheckpoint-th token; the backward
 * recomputes the states of one block of tokens from there (bit for bit, the
 * same operations) and walks that block from its last token to its first. */
static void bwd_job(void *vctx, int64_t job) {
  const bwd_ctx *c = (const bwd_ctx *)vctx;
  const int s = (int)(job / c->Hqk), qh = (int)(job % c->Hqk);
  const int K = c->K, V = c->V, G = c->Hv / c->Hqk, Hv = c->Hv, Hqk = c->Hqk;
  const int64_t t0 = c->cu[s], n = c->cu[s + 1] - t0, VK = (int64_t)V * K;
  const int64_t n_ck = n / kCheckpoint + 1;
  double *ck = (double *)malloc(sizeof(double) * n_ck * VK);
  double *st = (double *)malloc(sizeof(double) * (kCheckpoint + 1) * VK);
  double *dS = (double *)malloc(sizeof(double) * VK);
  double *qn = (double *)malloc(sizeof(double) * (n > 0 ? n : 1) * K);
  double *kn = (double *)malloc(sizeof(double) * (n > 0 ? n : 1) * K);
  double *dqn = (double *)calloc((size_t)(n > 0 ? n : 1) * K, sizeof(double));
  double *dkn = (double *)calloc((size_t)(n > 0 ? n : 1) * K, sizeof(double));
  double *r = (double *)malloc(sizeof(double) * V), *dr = (double *)malloc(sizeof(double) * V);
  double *dSk = (double *)malloc(sizeof(double) * V);
  for (int64_t i = 0; i < n; ++i) {
    const double *qraw = c->q + ((t0 + i) * Hqk + qh) * K, *kraw = c->k + ((t0 + i) * Hqk + qh) * K;
    if (c->l2norm) {
      l2_normalise(qraw, K, c->eps, qn + i * K);
      l2_normalise(kraw, K, c->eps, kn + i * K);
    } else {
      memcpy(qn + i * K, qraw, sizeof(double) * K);
      memcpy(kn + i * K, kraw, sizeof(double) * K);
    }
  }
  for (int hh = 0; hh < G; ++hh) {
    const int h = qh * G + hh;
    /* forward, keeping the checkpoints */
    if (c->h0) memcpy(st, c->h0 + ((int64_t)s * Hv + h) * VK, sizeof(double) * VK);
    else memset(st, 0, sizeof(double) * VK);
    for (int64_t i = 0; i < n; ++i) {
      if (i % kCheckpoint == 0) memcpy(ck + (i / kCheckpoint) * VK, st, sizeof(double) * VK);
      const int64_t t = t0 + i;
      fwd_token(st, kn + i * K, c->v + (t * Hv + h) * V, exp(c->g[t * Hv + h]), c->beta[t * Hv + h], K, V);
    }
    if (c->dhT) memcpy(dS, c->dhT + ((int64_t)s * Hv + h) * VK, sizeof(double) * VK);
    else memset(dS, 0, sizeof(double) * VK);
    for (int64_t b = (n - 1) / kCheckpoint; n > 0 && b >= 0; --b) {
      const int64_t i0 = b * kCheckpoint, i1 = (i0 + kCheckpoint < n) ? i0 + kCheckpoint : n;
      memcpy(st, ck + b * VK, sizeof(double) * VK); /* st[m] = state before token i0 + m */
      for (int64_t i = i0; i < i1; ++i) {
        const int64_t t = t0 + i;
        double *nx = st + (i - i0 + 1) * VK;
        memcpy(nx, nx - VK, sizeof(double) * VK);
        fwd_token(nx, kn + i * K, c->v + (t * Hv + h) * V, exp(c->g[t * Hv + h]), c->beta[t * Hv + h], K, V);
      }
      for (int64_t i = i1 - 1; i >= i0; --i) {
        const int64_t t = t0 + i;
        const double *Sp = st + (i - i0) * VK, *Sn = Sp + VK;
        const double *qt = qn + i * K, *kt = kn + i * K;
        const double *vt = c->v + (t * Hv + h) * V, *dot = c->dout + (t * Hv + h) * V;
        const double alpha = exp(c->g[t * Hv + h]), bt = c->beta[t * Hv + h];
        double *dqt = dqn + i * K, *dkt = dkn + i * K;
        /* o_t = scale S_t q */
        for (int a = 0; a < V; ++a)
          for (int j = 0; j < K; ++j) {
            dqt[j] += c->scale * Sn[(int64_t)a * K + j] * dot[a];
            dS[(int64_t)a * K + j] += c->scale * dot[a] * qt[j];
          }
        /* S_t = P + beta r k^T, r = v - P k, P = alpha S_{t-1} */
        double db = 0.0;
        for (int a = 0; a < V; ++a) {
          double pk = 0.0, sk = 0.0;
          for (int j = 0; j < K; ++j) {
            pk += (Sp[(int64_t)a * K + j] * alpha) * kt[j];
            sk += dS[(int64_t)a * K + j] * kt[j];
          }
          r[a] = vt[a] - pk;
          dSk[a] = sk;
          db += r[a] * sk;
        }
        for (int a = 0; a < V; ++a) {
          dr[a] = bt * dSk[a];
          c->dv[(t * Hv + h) * V + a] = dr[a];
        }
        for (int j = 0; j < K; ++j) {
          double acc = 0.0;
          for (int a = 0; a < V; ++a)
            acc += bt * dS[(int64_t)a * K + j] * r[a] - alpha * Sp[(int64_t)a * K + j] * dr[a];
          dkt[j] += acc;
        }
        double dalpha = 0.0;
        for (int a = 0; a < V; ++a)
          for (int j = 0; j < K; ++j) {
            const double dp = dS[(int64_t)a * K + j] - dr[a] * kt[j];
            dalpha += Sp[(int64_t)a * K + j] * dp;
            dS[(int64_t)a * K + j] = alpha * dp;
          }
        c->dg[t * Hv + h] = alpha * dalpha;
        c->dbeta[t * Hv + h] = db;
      }
    }
    if (c->dh0) memcpy(c->dh0 + ((int64_t)s * Hv + h) * VK, dS, sizeof(double) * VK);
  }
  for (int64_t i = 0; i < n; ++i) { /* back to the raw q and k */
    const int64_t off = ((t0 + i) * Hqk + qh) * K;
    if (c->l2norm) {
      l2_backward(c->q + off, dqn + i * K, K, c->eps, c->dq + off);
      l2_backward(c->k + off, dkn + i * K, K, c->eps, c->dk + off);
    } else {
      memcpy(c->dq + off, dqn + i * K, sizeof(double) * K);
      memcpy(c->dk + off, dkn + i * K, sizeof(double) * K);
    }
  }
  free(ck); free(st); free(dS); free(qn); free(kn); free(dqn); free(dkn); free(r); free(dr); free(dSk);
}

/* Gradients of every input for upstream dout [n_tok, Hv, V] and dhT (may be
 * NULL: no loss on the final state).  h0 may be NULL (zero start state); dh0
 * may be NULL.  Outputs have the layouts of the inputs. */
void oracle_gdn_bwd(const double *q, const double *k, const double *v, const double *g,
                    const double *beta, const double *h0, const int32_t *cu, int n_seq, int Hqk,
                    int Hv, int K, int V, double scale, int l2norm, double eps,
                    const double *dout, const double *dhT, double *dq, double *dk, double *dv,
                    double *dg, double *dbeta, double *dh0, int n_threads) {
  bwd_ctx c = {q, k, v, g, beta, h0, dout, dhT, cu, n_seq, Hqk, Hv, K, V, l2norm, scale, eps,
               dq, dk, dv, dg, dbeta, dh0};
  run_jobs(bwd_job, &c, (int64_t)n_seq * Hqk, n_threads);
}

/* -------------------------------------------------- segment summaries */

typedef struct {
  const double *k, *v, *g, *beta;
  const int32_t *bounds;
  int n_seg, Hqk, Hv, K, V, l2norm;
  double eps;
  double *M, *S_local;
} seg_ctx;

/* For segment [bounds[i], bounds[i+1]) and v-head h ("Qwen3.5 cp - #1",
 * Architecture and Patches: the (b, M) pair, M being the segment's total
 * transition), so that for ANY start state S_start
 *     S_end = S_start * M + S_local.
 *   M       = A_1 A_2 ... A_n,  A_t = exp(g_t) (I - beta_t k_t k_t^T)  (K x K)
 *   S_local = the state reached from S = 0 over the segment          (V x K)
 * M is accumulated as M <- M A_t; M (I - beta k k^T) is written as the
 * rank-1 update M - beta (M k) k^T, which is the same product. */
static void seg_job(void *vctx, int64_t job) {
  const seg_ctx *c = (const seg_ctx *)vctx;
  const int i = (int)(job / c->Hv), h = (int)(job % c->Hv);
  const int K = c->K, V = c->V, qh = h / (c->Hv / c->Hqk);
  double *M = c->M + ((int64_t)i * c->Hv + h) * K * K;
  double *S = c->S_local + ((int64_t)i * c->Hv + h) * V * K;
  double *kt = (double *)malloc(sizeof(double) * K);
  memset(M, 0, sizeof(double) * K * K);
  for (int a = 0; a < K; ++a) M[(int64_t)a * K + a] = 1.0;
  memset(S, 0, sizeof(double) * V * K);
  for (int64_t t = c->bounds[i]; t < c->bounds[i + 1]; ++t) {
    const double *kraw = c->k + (t * c->Hqk + qh) * K;
    if (c->l2norm) l2_normalise(kraw, K, c->eps, kt);
    else memcpy(kt, kraw, sizeof(double) * K);
    const double alpha = exp(c->g[t * c->Hv + h]);
    const double bt = c->beta[t * c->Hv + h];
    const double *vt = c->v + (t * c->Hv + h) * V;
    for (int a = 0; a < K; ++a) { /* M <- M A_t, row by row */
      double *row = M + (int64_t)a * K;
      double mk = 0.0;
      for (int j = 0; j < K; ++j) mk += row[j] * kt[j];
      for (int j = 0; j < K; ++j) row[j] = alpha * (row[j] - bt * mk * kt[j]);
    }
    for (int a = 0; a < V; ++a) { /* S <- S A_t + beta v k^T */
      double *row = S + (int64_t)a * K;
      double sk = 0.0;
      for (int j = 0; j < K; ++j) sk += row[j] * kt[j];
      for (int j = 0; j < K; ++j)
        row[j] = alpha * (row[j] - bt * sk * kt[j]) + bt * vt[a] * kt[j];
    }
  }
  free(kt);
}

void oracle_segment_summary(const double *k, const double *v, const double *g,
                            const double *beta, const int32_t *bounds, int n_seg,
                            int Hqk, int Hv, int K, int V, int l2norm, double eps,
                            double *M, double *S_local, int n_threads) {
  seg_ctx c = {k, v, g, beta, bounds, n_seg, Hqk, Hv, K, V, l2norm, eps, M, S_local};
  run_jobs(seg_job, &c, (int64_t)n_seg * Hv, n_threads);
}

/* Chain reduce ("Qwen3.5 cp - #1", Architecture: (b, M) chain reduce):
 *   S_start[0] = h0 (or 0);  S_start[i+1] = S_start[i] M_i + S_local[i];
 *   hT = S_start[n_seg]. */
void oracle_chain_reduce(const double *M, const double *S_local,
                         const double *h0, int n_seg, int Hv, int K, int V,
                         double *S_start, double *hT) {
  double *S = (double *)malloc(sizeof(double) * V * K);
  double *nxt = (double *)malloc(sizeof(double) * V * K);
  for (int h = 0; h < Hv; ++h) {
    if (h0) memcpy(S, h0 + (int64_t)h * V * K, sizeof(double) * V * K);
    else memset(S, 0, sizeof(double) * V * K);
    for (int i = 0; i < n_seg; ++i) {
      const double *Mi = M + ((int64_t)i * Hv + h) * K * K;
      const double *Li = S_local + ((int64_t)i * Hv + h) * V * K;
      memcpy(S_start + ((int64_t)i * Hv + h) * V * K, S, sizeof(double) * V * K);
      for (int a = 0; a < V; ++a) {
        for (int j = 0; j < K; ++j) {
          double acc = Li[(int64_t)a * K + j];
          for (int m = 0; m < K; ++m) acc += S[(int64_t)a * K + m] * Mi[(int64_t)m * K + j];
          nxt[(int64_t)a * K + j] = acc;
        }
      }
      memcpy(S, nxt, sizeof(double) * V * K);
    }
    if (hT) memcpy(hT + (int64_t)h * V * K, S, sizeof(double) * V * K);
  }
  free(S);
  free(nxt);
}

/* cu_seqlens from position_ids ("[v1] support GDN Ulysses cp", Key decisions
 * 4): a new sample starts at token 0 and wherever position_ids returns to 0.
 * Writes n_seq+1 offsets into cu (room for n_tok+1) and returns n_seq. */
int oracle_cu_seqlens_from_position_ids(const int64_t *pos, int64_t n_tok, int32_t *cu) {
  int n = 0;
  for (int64_t t = 0; t < n_tok; ++t)
    if (t == 0 || pos[t] == 0) cu[n++] = (int32_t)t;
  cu[n] = (int32_t)n_tok;
  return n_tok == 0 ? 0 : n;
}
