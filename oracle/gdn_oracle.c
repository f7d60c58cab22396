/*
 * Float64 oracle of the gated delta-rule linear-attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code with the CUDA path.
 *
 * Source: "Qwen3.5-9B-npu" model card, section "How it works":
 *   - the per-token gated delta rule (the four-line recurrence over a
 *     per-head [128 x 128] state): gdn_oracle_recurrent();
 *   - the chunkwise-parallel prompt-block form (G = cumsum(g), strictly
 *     lower N, per-token deltas D, block output O, carried state S_T),
 *     with partly filled blocks padded by g = 0, beta = 0 tokens, and the
 *     triangular inverse by forward substitution or by exact block
 *     doubling: gdn_oracle_chunked(), gdn_oracle_tril_inverse().
 *
 * All arithmetic is in double.  Inputs are float32 arrays (bfloat16 inputs
 * are widened exactly by the caller), so the oracle sees exactly the
 * values the GPU sees.
 *
 * Layouts (row-major, contiguous):
 *   q, k        [T, Hk, dk]        v, o   [T, Hv, dv]
 *   g, beta     [T, Hv]            state  [N, Hv, dk, dv]  (S[i][j]: i key, j value)
 *   cu_seqlens  [N + 1]
 * v-head h reads q/k head h / (Hv / Hk).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int num_seqs, hk, hv, dk, dv;
  const int32_t *cu_seqlens;
  const float *q, *k, *v, *g, *beta, *state_in;
  double *o, *state_out;
  const int32_t *pairs;  /* 2 * num_chains ints (n, h), or NULL for all */
  int num_chains;
  int chunk;             /* chunked form only */
  int solve;             /* 0: forward substitution, 1: block doubling */
  int next;              /* shared work counter */
  int err;
  double *delta_out;     /* per-token deltas [T, Hv, dv], or NULL */
} job_t;

static void chain_of(const job_t *J, int idx, int *n, int *h) {
  if (J->pairs) {
    *n = J->pairs[2 * idx];
    *h = J->pairs[2 * idx + 1];
  } else {
    *n = idx / J->hv;
    *h = idx % J->hv;
  }
}

static void load_state(const job_t *J, int n, int h, double *S) {
  size_t sz = (size_t)J->dk * J->dv;
  if (J->state_in) {
    const float *src = J->state_in + ((size_t)n * J->hv + h) * sz;
    for (size_t e = 0; e < sz; ++e) S[e] = (double)src[e];
  } else {
    memset(S, 0, sz * sizeof(double));
  }
}

static void store_state(const job_t *J, int n, int h, const double *S) {
  size_t sz = (size_t)J->dk * J->dv;
  memcpy(J->state_out + ((size_t)n * J->hv + h) * sz, S, sz * sizeof(double));
}

/* ------------------------------------------------------------------ *
 * Per-token recurrence, in the order the page gives it:               *
 *   S <- S * exp(g_t); kv <- S^T k_t; S <- S + k_t (x) ((v_t - kv)    *
 *   * beta_t); o_t <- S^T q_t  (the output reads the updated state).  *
 * ------------------------------------------------------------------ */
static void recurrent_chain(const job_t *J, int n, int h, double *S, double *kv,
                            double *delta) {
  const int dk = J->dk, dv = J->dv, hk = J->hk, hv = J->hv;
  const int kh = h / (hv / hk);
  load_state(J, n, h, S);
  for (int t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
    const float *qt = J->q + ((size_t)t * hk + kh) * dk;
    const float *kt = J->k + ((size_t)t * hk + kh) * dk;
    const float *vt = J->v + ((size_t)t * hv + h) * dv;
    const double decay = exp((double)J->g[(size_t)t * hv + h]);
    const double b = (double)J->beta[(size_t)t * hv + h];
    for (int e = 0; e < dk * dv; ++e) S[e] *= decay;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[i * dv + j] * (double)kt[i];
      kv[j] = acc;
    }
    for (int j = 0; j < dv; ++j) delta[j] = ((double)vt[j] - kv[j]) * b;
    if (J->delta_out) memcpy(J->delta_out + ((size_t)t * hv + h) * dv, delta, sizeof(double) * dv);
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += (double)kt[i] * delta[j];
    double *ot = J->o + ((size_t)t * hv + h) * dv;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[i * dv + j] * (double)qt[i];
      ot[j] = acc;
    }
  }
  store_state(J, n, h, S);
}

/* ------------------------------------------------------------------ *
 * Inverse of the unit lower-triangular matrix M = I + Nm (n x n).      *
 * method 0: forward substitution, column by column.                    *
 * method 1: exact block doubling.  Diagonal blocks of size b are       *
 *   inverted first (b = 1: the unit diagonal); two neighbouring blocks *
 *   P (top) and R (bottom) with the block Q below P combine by         *
 *   (D + C)^-1 = D^-1 - D^-1 C D^-1, D = diag(P, R), C = [[0,0],[Q,0]], *
 *   i.e. the new lower-left block is -R^-1 Q P^-1.  Every intermediate *
 *   is the inverse of a leading diagonal sub-block.                    *
 * ------------------------------------------------------------------ */
static void tril_inverse(int n, const double *Nm, double *X, int method, double *tmp) {
  memset(X, 0, (size_t)n * n * sizeof(double));
  if (method == 0) {
    for (int c = 0; c < n; ++c) {
      /* solve (I + Nm) x = e_c */
      for (int r = 0; r < n; ++r) {
        double acc = (r == c) ? 1.0 : 0.0;
        for (int j = 0; j < r; ++j) acc -= Nm[r * n + j] * X[j * n + c];
        X[r * n + c] = acc;
      }
    }
    return;
  }
  for (int i = 0; i < n; ++i) X[i * n + i] = 1.0;
  for (int b = 1; b < n; b *= 2) {
    for (int p0 = 0; p0 + b < n; p0 += 2 * b) {
      const int r0 = p0 + b;                      /* first row of R */
      const int rb = (r0 + b <= n) ? b : n - r0;  /* size of R */
      /* tmp = Q P^-1, Q = rows r0.., cols p0.. of M (= Nm there) */
      for (int r = 0; r < rb; ++r)
        for (int c = 0; c < b; ++c) {
          double acc = 0.0;
          for (int m = 0; m < b; ++m)
            acc += Nm[(r0 + r) * n + (p0 + m)] * X[(p0 + m) * n + (p0 + c)];
          tmp[r * b + c] = acc;
        }
      /* X[R rows, P cols] = -R^-1 (Q P^-1) */
      for (int r = 0; r < rb; ++r)
        for (int c = 0; c < b; ++c) {
          double acc = 0.0;
          for (int m = 0; m < rb; ++m) acc += X[(r0 + r) * n + (r0 + m)] * tmp[m * b + c];
          X[(r0 + r) * n + (p0 + c)] = -acc;
        }
    }
  }
}

/* ------------------------------------------------------------------ *
 * Chunkwise-parallel form over blocks of C tokens.  With G the         *
 * inclusive cumsum of g inside the block and S0 the incoming state:    *
 *   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t}                    *
 *   D   = (I + N)^-1 diag(beta) (V - diag(exp G) K S0)                 *
 *   O   = diag(exp G) Q S0 + [exp(G_t - G_j) q_t.k_j]_{j<=t} D         *
 *   S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D                       *
 * A block that runs past the sequence end is padded with tokens of     *
 * g = 0, beta = 0 (and q = k = v = 0), which leave the state as it was. *
 * ------------------------------------------------------------------ */
typedef struct {
  double *S, *G, *b, *K, *Q, *V, *Nm, *A, *Tinv, *R, *D, *tmp;
} chunk_ws;

static void chunked_chain(const job_t *J, int n, int h, chunk_ws *w) {
  const int dk = J->dk, dv = J->dv, hk = J->hk, hv = J->hv, C = J->chunk;
  const int kh = h / (hv / hk);
  double *S = w->S;
  load_state(J, n, h, S);
  const int bos = J->cu_seqlens[n], eos = J->cu_seqlens[n + 1];
  for (int c0 = bos; c0 < eos; c0 += C) {
    /* gather the block, padding past eos */
    double gsum = 0.0;
    for (int t = 0; t < C; ++t) {
      const int tok = c0 + t;
      const int valid = tok < eos;
      const double gt = valid ? (double)J->g[(size_t)tok * hv + h] : 0.0;
      w->b[t] = valid ? (double)J->beta[(size_t)tok * hv + h] : 0.0;
      gsum += gt;
      w->G[t] = gsum;
      for (int i = 0; i < dk; ++i) {
        w->K[t * dk + i] = valid ? (double)J->k[((size_t)tok * hk + kh) * dk + i] : 0.0;
        w->Q[t * dk + i] = valid ? (double)J->q[((size_t)tok * hk + kh) * dk + i] : 0.0;
      }
      for (int j = 0; j < dv; ++j)
        w->V[t * dv + j] = valid ? (double)J->v[((size_t)tok * hv + h) * dv + j] : 0.0;
    }
    /* N (strictly lower) and the decay-masked causal A (lower, with diagonal) */
    for (int t = 0; t < C; ++t)
      for (int j = 0; j < C; ++j) {
        double kk = 0.0, qk = 0.0;
        for (int i = 0; i < dk; ++i) {
          kk += w->K[t * dk + i] * w->K[j * dk + i];
          qk += w->Q[t * dk + i] * w->K[j * dk + i];
        }
        const double decay = exp(w->G[t] - w->G[j]);
        w->Nm[t * C + j] = (j < t) ? w->b[t] * decay * kk : 0.0;
        w->A[t * C + j] = (j <= t) ? decay * qk : 0.0;
      }
    /* R = diag(beta) (V - diag(exp G) K S0) */
    for (int t = 0; t < C; ++t)
      for (int j = 0; j < dv; ++j) {
        double ks = 0.0;
        for (int i = 0; i < dk; ++i) ks += w->K[t * dk + i] * S[i * dv + j];
        w->R[t * dv + j] = w->b[t] * (w->V[t * dv + j] - exp(w->G[t]) * ks);
      }
    /* D = (I + N)^-1 R */
    tril_inverse(C, w->Nm, w->Tinv, J->solve, w->tmp);
    for (int t = 0; t < C; ++t)
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int m = 0; m <= t; ++m) acc += w->Tinv[t * C + m] * w->R[m * dv + j];
        w->D[t * dv + j] = acc;
      }
    /* O = diag(exp G) Q S0 + A D, for the valid rows */
    for (int t = 0; t < C && c0 + t < eos; ++t) {
      double *ot = J->o + ((size_t)(c0 + t) * hv + h) * dv;
      for (int j = 0; j < dv; ++j) {
        double qs = 0.0, ad = 0.0;
        for (int i = 0; i < dk; ++i) qs += w->Q[t * dk + i] * S[i * dv + j];
        for (int m = 0; m <= t; ++m) ad += w->A[t * C + m] * w->D[m * dv + j];
        ot[j] = exp(w->G[t]) * qs + ad;
      }
    }
    /* S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D */
    const double GT = w->G[C - 1];
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int t = 0; t < C; ++t) acc += w->K[t * dk + i] * exp(GT - w->G[t]) * w->D[t * dv + j];
        S[i * dv + j] = exp(GT) * S[i * dv + j] + acc;
      }
  }
  store_state(J, n, h, S);
}

/* ------------------------------------------------------------------ threads */

static void *recurrent_worker(void *arg) {
  job_t *J = (job_t *)arg;
  double *S = malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double *kv = malloc(sizeof(double) * J->dv);
  double *delta = malloc(sizeof(double) * J->dv);
  if (!S || !kv || !delta) {
    __atomic_store_n(&J->err, 1, __ATOMIC_SEQ_CST);
  } else {
    for (;;) {
      int idx = __atomic_fetch_add(&J->next, 1, __ATOMIC_SEQ_CST);
      if (idx >= J->num_chains) break;
      int n, h;
      chain_of(J, idx, &n, &h);
      recurrent_chain(J, n, h, S, kv, delta);
    }
  }
  free(S);
  free(kv);
  free(delta);
  return NULL;
}

static void *chunked_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const size_t C = J->chunk, dk = J->dk, dv = J->dv;
  chunk_ws w;
  w.S = malloc(sizeof(double) * dk * dv);
  w.G = malloc(sizeof(double) * C);
  w.b = malloc(sizeof(double) * C);
  w.K = malloc(sizeof(double) * C * dk);
  w.Q = malloc(sizeof(double) * C * dk);
  w.V = malloc(sizeof(double) * C * dv);
  w.Nm = malloc(sizeof(double) * C * C);
  w.A = malloc(sizeof(double) * C * C);
  w.Tinv = malloc(sizeof(double) * C * C);
  w.R = malloc(sizeof(double) * C * dv);
  w.D = malloc(sizeof(double) * C * dv);
  w.tmp = malloc(sizeof(double) * C * C);
  if (!w.S || !w.G || !w.b || !w.K || !w.Q || !w.V || !w.Nm || !w.A || !w.Tinv || !w.R ||
      !w.D || !w.tmp) {
    __atomic_store_n(&J->err, 1, __ATOMIC_SEQ_CST);
  } else {
    for (;;) {
      int idx = __atomic_fetch_add(&J->next, 1, __ATOMIC_SEQ_CST);
      if (idx >= J->num_chains) break;
      int n, h;
      chain_of(J, idx, &n, &h);
      chunked_chain(J, n, h, &w);
    }
  }
  free(w.S); free(w.G); free(w.b); free(w.K); free(w.Q); free(w.V);
  free(w.Nm); free(w.A); free(w.Tinv); free(w.R); free(w.D); free(w.tmp);
  return NULL;
}

static int run(job_t *J, void *(*worker)(void *), int threads) {
  if (J->num_seqs < 0 || J->hk <= 0 || J->hv <= 0 || J->hv % J->hk || J->dk <= 0 ||
      J->dv <= 0)
    return 1;
  if (!J->pairs) J->num_chains = J->num_seqs * J->hv;
  if (threads < 1) threads = 1;
  if (threads > J->num_chains) threads = J->num_chains > 0 ? J->num_chains : 1;
  J->next = 0;
  J->err = 0;
  pthread_t *tid = malloc(sizeof(pthread_t) * threads);
  if (!tid) return 1;
  int started = 0;
  for (int i = 1; i < threads; ++i) {
    if (pthread_create(&tid[i], NULL, worker, J) != 0) break;
    started = i;
  }
  worker(J);
  for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
  free(tid);
  return J->err;
}

/* ------------------------------------------------------------------ API */

/* Per-token recurrence over every (sequence, v-head) chain, or over the
 * `num_pairs` chains listed in `pairs` (n, h pairs).  Writes o rows and
 * state_out blocks of the chains it runs; other entries are untouched.
 * state_in may be NULL (zero initial state).  Returns 0 on success. */
int gdn_oracle_recurrent(int num_seqs, int hk, int hv, int dk, int dv,
                         const int32_t *cu_seqlens, const float *q, const float *k,
                         const float *v, const float *g, const float *beta,
                         const float *state_in, double *o, double *state_out,
                         const int32_t *pairs, int num_pairs, int threads) {
  job_t J = {num_seqs, hk, hv, dk, dv, cu_seqlens, q, k, v, g, beta, state_in, o, state_out,
             pairs, num_pairs, 0, 0, 0, 0, NULL};
  return run(&J, recurrent_worker, threads);
}

/* The same recurrence, also writing each token's delta
 *   delta_t = (v_t - S'^T k_t) * beta_t      (S' the decayed state before the write)
 * to delta_out [T, Hv, dv]: the rows D of the chunkwise form ("How it works": the
 * per-token deltas), from which the state after any prefix of a block follows. */
int gdn_oracle_recurrent_deltas(int num_seqs, int hk, int hv, int dk, int dv,
                                const int32_t *cu_seqlens, const float *q, const float *k,
                                const float *v, const float *g, const float *beta,
                                const float *state_in, double *o, double *state_out,
                                double *delta_out, int threads) {
  job_t J = {num_seqs, hk, hv, dk, dv, cu_seqlens, q, k, v, g, beta, state_in, o, state_out,
             NULL, 0, 0, 0, 0, 0, delta_out};
  return run(&J, recurrent_worker, threads);
}

/* Chunkwise-parallel form with block length `chunk`; `solve` selects the
 * triangular inverse (0 forward substitution, 1 block doubling). */
int gdn_oracle_chunked(int num_seqs, int hk, int hv, int dk, int dv, const int32_t *cu_seqlens,
                       const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const float *state_in, double *o, double *state_out,
                       const int32_t *pairs, int num_pairs, int chunk, int solve, int threads) {
  if (chunk <= 0) return 1;
  job_t J = {num_seqs, hk, hv, dk, dv, cu_seqlens, q, k, v, g, beta, state_in, o, state_out,
             pairs, num_pairs, chunk, solve, 0, 0, NULL};
  return run(&J, chunked_worker, threads);
}

/* X = (I + Nm)^-1 for a strictly lower-triangular n x n Nm (entries on and
 * above the diagonal are ignored).  method 0: forward substitution,
 * method 1: block doubling.  Returns 0 on success. */
int gdn_oracle_tril_inverse(int n, const double *Nm, double *X, int method) {
  if (n <= 0) return 1;
  double *lower = calloc((size_t)n * n, sizeof(double));
  double *tmp = malloc(sizeof(double) * (size_t)n * n);
  if (!lower || !tmp) {
    free(lower);
    free(tmp);
    return 1;
  }
  for (int r = 0; r < n; ++r)
    for (int c = 0; c < r; ++c) lower[r * n + c] = Nm[r * n + c];
  tril_inverse(n, lower, X, method, tmp);
  free(lower);
  free(tmp);
  return 0;
}

/* ---------------------------------------------------------------------------
 * The GDN block around the recurrence.  "Qwen3.5-4B — Hexagon NPU (QHexRT) — v81"
 * model card, introduction: each linear-attention layer is a short causal-conv FIFO +
 * the recurrent (SSM) state + a gated RMSNorm; "Qwen3.5-0.8B on Dragon Q6A NPU via QNN
 * EP", main changes: the gates use Softplus; "Qwen3.5-9B-npu", "How it works": the output
 * only feeds the scale-invariant gated RMSNorm.  The pages give no formulas for these
 * steps; the readings taken are stated at each function.
 */

static double silu_d(double u) { return u / (1.0 + exp(-u)); }
static double softplus_d(double u) { return u > 0.0 ? u + log1p(exp(-u)) : log1p(exp(u)); }

/* Input prologue.  For sequence n (tokens [cu[n], cu[n+1]); cu_seqlens == NULL: token n
 * alone) and channel c of the concatenated raw projections
 *   x = [q_raw (hk*dk) | k_raw (hk*dk) | v_raw (hv*dv)]:
 *   y_t[c] = SiLU( sum_{i=0}^{W-1} w[c][i] * x_{t-(W-1)+i}[c] ),   W = conv_width,
 * where x_p before the sequence's first token is conv_state_in[n][c][p - bos + W - 1]
 * (the FIFO of the W-1 raw inputs before the call; zero when conv_state_in is NULL) and
 * SiLU(u) = u / (1 + e^-u).  The q and k rows are then L2-normalised per (token, head):
 * y / sqrt(sum y^2 + eps).  Gates per (token, v-head):
 *   g = -exp(A_log[h]) softplus(a + dt_bias[h]),  beta = 1 / (1 + e^-b),
 * softplus(u) = log(1 + e^u).  conv_state_out[n][c][j] = x_{eos-(W-1)+j}: the FIFO advanced
 * by the sequence's tokens.  Returns 0 on success. */
int gdn_oracle_prologue(int num_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                        int conv_width, const int32_t *cu_seqlens, const float *q_raw,
                        const float *k_raw, const float *v_raw, const float *a, const float *b,
                        const float *conv_w, const float *A_log, const float *dt_bias,
                        const float *conv_state_in, double eps, double *q, double *k, double *v,
                        double *g, double *beta, double *conv_state_out) {
  const int W = conv_width, cq = hk * dk, cv = hv * dv, ch = 2 * cq + cv;
  if (W < 1 || num_seqs < 0 || total_tokens < 0) return 1;
  double *y = malloc(sizeof(double) * (size_t)(ch > 0 ? ch : 1));
  if (!y) return 1;
  for (int n = 0; n < num_seqs; ++n) {
    const int bos = cu_seqlens ? cu_seqlens[n] : n, eos = cu_seqlens ? cu_seqlens[n + 1] : n + 1;
    for (int t = bos; t < eos; ++t) {
      for (int c = 0; c < ch; ++c) {
        double acc = 0.0;
        for (int i = 0; i < W; ++i) {
          const int p = t - (W - 1) + i;
          double xv;
          if (p >= bos) {
            xv = c < cq ? q_raw[(size_t)p * cq + c]
               : c < 2 * cq ? k_raw[(size_t)p * cq + (c - cq)] : v_raw[(size_t)p * cv + (c - 2 * cq)];
          } else {
            xv = conv_state_in ? conv_state_in[((size_t)n * ch + c) * (W - 1) + (p - bos + W - 1)] : 0.0;
          }
          acc += (double)conv_w[(size_t)c * W + i] * xv;
        }
        y[c] = silu_d(acc);
      }
      for (int hd = 0; hd < 2 * hk; ++hd) {  /* q heads, then k heads */
        double ss = 0.0;
        for (int i = 0; i < dk; ++i) ss += y[hd * dk + i] * y[hd * dk + i];
        const double sc = 1.0 / sqrt(ss + eps);
        double *dst = hd < hk ? q + ((size_t)t * hk + hd) * dk : k + ((size_t)t * hk + hd - hk) * dk;
        for (int i = 0; i < dk; ++i) dst[i] = y[hd * dk + i] * sc;
      }
      for (int j = 0; j < cv; ++j) v[(size_t)t * cv + j] = y[2 * cq + j];
      for (int h = 0; h < hv; ++h) {
        const size_t gi = (size_t)t * hv + h;
        g[gi] = -exp((double)A_log[h]) * softplus_d((double)a[gi] + (double)dt_bias[h]);
        beta[gi] = 1.0 / (1.0 + exp(-(double)b[gi]));
      }
    }
    for (int c = 0; c < ch; ++c)
      for (int j = 0; j < W - 1; ++j) {
        const int p = eos - (W - 1) + j;
        double xv;
        if (p >= bos) {
          xv = c < cq ? q_raw[(size_t)p * cq + c]
             : c < 2 * cq ? k_raw[(size_t)p * cq + (c - cq)] : v_raw[(size_t)p * cv + (c - 2 * cq)];
        } else {
          xv = conv_state_in ? conv_state_in[((size_t)n * ch + c) * (W - 1) + (p - bos + W - 1)] : 0.0;
        }
        conv_state_out[((size_t)n * ch + c) * (W - 1) + j] = xv;
      }
  }
  free(y);
  return 0;
}

/* Output epilogue, the gated RMSNorm of each (token, v-head) row of d values:
 *   y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z),
 * with one weight vector [d] shared by every head.  Returns 0 on success. */
int gdn_oracle_gated_rmsnorm(int rows, int d, const float *o, const float *z, const float *weight,
                             double eps, double *y) {
  if (rows < 0 || d <= 0) return 1;
  for (int r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += (double)o[(size_t)r * d + i] * o[(size_t)r * d + i];
    const double sc = 1.0 / sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i)
      y[(size_t)r * d + i] = o[(size_t)r * d + i] * sc * weight[i] * silu_d(z[(size_t)r * d + i]);
  }
  return 0;
}
