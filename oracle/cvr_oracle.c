/* CPU oracle of the CVR scoring forward pass -- TEST INFRASTRUCTURE (see cvr_oracle.h).
 *
 * Sources of each step (page title abbreviated; "iQIYI CVR" is the article
 * "爱奇艺广告CVR模型参数量10倍增长 ..." at m.bobobaike.com/news/370088.html and
 * "GPU CTR inference" is "广告 CTR 预估模型的 GPU 推理优化" at gtnt.cn/news/20674):
 *   pooling        iQIYI CVR 3.1 (item 2: multi-valued features aggregate by mean, not sum)
 *   clamp, cast    GPU CTR inference 三 (clamp to [-10, 10] after the lookup, then half precision)
 *   inputs         iQIYI CVR 3.2.1 (sequence events concat 4 embedded columns; non-sequence
 *                  fields concat; three groups share one id table)
 *   tokens         iQIYI CVR 3.2.2 / 3.2.3 (non-sequence embedding split into N heads/tokens;
 *                  each sequence through its own SwiGLU)
 *   Query Decoding iQIYI CVR 3.2.3 (per group one FFN query from the N tokens + the mean-pooled
 *                  sequence; K/V are the encoded states; temperature-scaled softmax)
 *   Query Boosting iQIYI CVR 3.2.3 (N+3 tokens, split -> mix -> revert, then residual)
 *   stacking       iQIYI CVR 3.2.3 (the interaction layer stacks like a decoder layer)
 *   prediction     iQIYI CVR 3.2.4 (PLE of 3 single-layer experts + two-layer heads per task)
 *   user/item      iQIYI CVR 3.4.5 (one user per request, many candidates, linked by request id)
 *
 * Where the pages leave a step open, the readings taken are listed beside the step.
 */
#include "cvr_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "../synth/cvr_synth.h"

/* ------------------------------------------------------------------------------------------ */
/* half-precision cast after the lookup (GPU CTR inference 三; bf16 per iQIYI CVR 3.4.3)       */
double oracle_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (double)x; /* Inf/NaN pass through */
  u += 0x7FFFu + ((u >> 16) & 1u);                        /* round to nearest, ties to even */
  u &= 0xFFFF0000u;
  float y;
  memcpy(&y, &u, 4);
  return (double)y;
}

static void table_row(const oracle_table* t, int64_t row, int32_t dim, float* out) {
  if (t->data) {
    memcpy(out, t->data + row * dim, (size_t)dim * sizeof(float));
  } else {
    for (int32_t c = 0; c < dim; ++c) out[c] = synth_table_value(t->seed, t->index, (uint64_t)row, (uint32_t)c,
                                                                (uint32_t)dim, t->scale);
  }
}

/* Mean-pooled embedding bag (iQIYI CVR 3.1 item 2) with the clamp of GPU CTR inference 三.
 * The sum runs in fp32, in bag order, from 0.0f; the mean is one IEEE division by the bag size;
 * the clamp is applied to the mean. An empty bag pools to zeros. An id outside [0, rows) reads
 * row 0 and makes the call return ORACLE_E_ID_RANGE. */
int oracle_pool_bag(const oracle_table* t, const int64_t* ids, int64_t n, int32_t dim, double clamp, float* out,
                    int64_t* rows_out) {
  int status = ORACLE_OK;
  float row[512];
  for (int32_t c = 0; c < dim; ++c) out[c] = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    int64_t id = ids[i];
    if (id < 0 || id >= t->rows) {
      id = 0;
      status = ORACLE_E_ID_RANGE;
    }
    if (rows_out) rows_out[i] = id;
    table_row(t, id, dim, row);
    for (int32_t c = 0; c < dim; ++c) out[c] = out[c] + row[c];
  }
  const float cl = (float)clamp;
  for (int32_t c = 0; c < dim; ++c) {
    float v = n > 0 ? out[c] / (float)n : 0.0f;
    if (v > cl) v = cl;
    if (v < -cl) v = -cl;
    out[c] = v;
  }
  return status;
}

/* ------------------------------------------------------------------------------------------ */
static double silu(double a) { return a / (1.0 + exp(-a)); }

/* y = W x + b for W [dout][din] (fp32 storage of bf16 values), x, y fp64. */
static void linear(const double* x, int32_t din, int32_t dout, const float* w, const float* b, double* y) {
  for (int32_t o = 0; o < dout; ++o) {
    double acc = b ? (double)b[o] : 0.0;
    const float* wr = w + (int64_t)o * din;
    for (int32_t i = 0; i < din; ++i) acc += (double)wr[i] * x[i];
    y[o] = acc;
  }
}

/* SwiGLU feed-forward: y = W2 (silu(W1 x + b1) * (W3 x + b3)) + b2 (iQIYI CVR 3.2.2: each
 * behaviour sequence is mapped position-wise by a SwiGLU network; sizes 128 -> 256 -> 128 from
 * the workload definitions; the Token Mixer of 3.2.3 uses the same form). */
void oracle_swiglu(const double* x, int32_t din, int32_t dh, int32_t dout, const float* w1, const float* b1,
                   const float* w3, const float* b3, const float* w2, const float* b2, double* y) {
  double* a = (double*)malloc(sizeof(double) * (size_t)dh * 3);
  double* g = a + dh;
  double* h = g + dh;
  linear(x, din, dh, w1, b1, a);
  linear(x, din, dh, w3, b3, g);
  for (int32_t j = 0; j < dh; ++j) h[j] = silu(a[j]) * g[j];
  linear(h, dh, dout, w2, b2, y);
  free(a);
}

/* Multi-head tokenisation (iQIYI CVR 3.2.2 / 3.2.3). The formula is missing from the page;
 * the reading taken is one linear map of the concatenated non-sequence embedding [user ; item]
 * to n_tokens * token_dim outputs, token n being outputs [n*token_dim, (n+1)*token_dim). */
void oracle_tokenize(const double* u, int32_t du, const double* it, int32_t di, const float* w, const float* b,
                     int32_t n_tokens, int32_t token_dim, double* x) {
  double* e = (double*)malloc(sizeof(double) * (size_t)(du + di));
  for (int32_t i = 0; i < du; ++i) e[i] = u[i];
  for (int32_t i = 0; i < di; ++i) e[du + i] = it[i];
  linear(e, du + di, n_tokens * token_dim, w, b, x);
  free(e);
}

/* Query construction (iQIYI CVR 3.2.3, Query Decoding item 1): the N non-sequence tokens and the
 * group's mean-pooled sequence vector are concatenated and passed through one FFN layer (read as a
 * single linear layer with bias, no activation) to give one query token per group. */
void oracle_query(const double* x, int32_t n_tokens, int32_t token_dim, const double* m_g, const float* w,
                  const float* b, double* q) {
  const int32_t din = (n_tokens + 1) * token_dim;
  double* in = (double*)malloc(sizeof(double) * (size_t)din);
  for (int32_t i = 0; i < n_tokens * token_dim; ++i) in[i] = x[i];
  for (int32_t i = 0; i < token_dim; ++i) in[n_tokens * token_dim + i] = m_g[i];
  linear(in, din, token_dim, w, b, q);
  free(in);
}

/* Cross-attention of one query over a group's encoded sequence (iQIYI CVR 3.2.3, Query Decoding
 * item 2 and the temperature remark): K = V = H (no projections), the query split into `heads`
 * heads of token_dim/heads, logits scaled by 1/(tau*sqrt(head_dim)), softmax over the sequence
 * (max-subtracted), output = concatenated per-head weighted sums of V. */
void oracle_cross_attention(const double* q, const double* H, int32_t L, int32_t token_dim, int32_t heads,
                            double tau, double* d, double* probs) {
  const int32_t dh = token_dim / heads;
  const double scale = 1.0 / (tau * sqrt((double)dh));
  double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  for (int32_t h = 0; h < heads; ++h) {
    double mx = -INFINITY;
    for (int32_t l = 0; l < L; ++l) {
      double acc = 0.0;
      for (int32_t i = 0; i < dh; ++i) acc += q[h * dh + i] * H[(int64_t)l * token_dim + h * dh + i];
      s[l] = acc * scale;
      if (s[l] > mx) mx = s[l];
    }
    double sum = 0.0;
    for (int32_t l = 0; l < L; ++l) {
      s[l] = exp(s[l] - mx);
      sum += s[l];
    }
    for (int32_t l = 0; l < L; ++l) s[l] /= sum;
    if (probs)
      for (int32_t l = 0; l < L; ++l) probs[h * L + l] = s[l];
    for (int32_t i = 0; i < dh; ++i) {
      double acc = 0.0;
      for (int32_t l = 0; l < L; ++l) acc += s[l] * H[(int64_t)l * token_dim + h * dh + i];
      d[h * dh + i] = L > 0 ? acc : 0.0;
    }
  }
  free(s);
}

/* Token Mixer split + mix (iQIYI CVR 3.2.3, Query Boosting; TokenMixer-Large): each of the T
 * tokens is split into T heads of D/T; mixed token j gathers head j of every token, token t's
 * head landing in slot t: mixed[j][t*hd + e] = z[t][j*hd + e]. */
void oracle_mix(const double* z, int32_t T, int32_t D, double* mixed) {
  const int32_t hd = D / T;
  for (int32_t j = 0; j < T; ++j)
    for (int32_t t = 0; t < T; ++t)
      for (int32_t e = 0; e < hd; ++e) mixed[j * D + t * hd + e] = z[t * D + j * hd + e];
}

/* Revert: the inverse index map of oracle_mix, back to the original token semantics. */
void oracle_revert(const double* mixed, int32_t T, int32_t D, double* z) {
  const int32_t hd = D / T;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t j = 0; j < T; ++j)
      for (int32_t e = 0; e < hd; ++e) z[t * D + j * hd + e] = mixed[j * D + t * hd + e];
}

/* RMSNorm: y = x * gain / sqrt(mean(x^2) + eps). */
void oracle_rmsnorm(const double* x, int32_t D, const float* gain, double eps, double* y) {
  double ss = 0.0;
  for (int32_t i = 0; i < D; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss / D + eps);
  for (int32_t i = 0; i < D; ++i) y[i] = x[i] * inv * (double)gain[i];
}

/* Query Boosting Token Mixer (iQIYI CVR 3.2.3): Y = RMSNorm(Z + Revert(F(Mix(Z)))), F a SwiGLU
 * shared by all mixed tokens; RMSNorm after the residual (post-norm) is the reading taken for the
 * normalisation that the workload definition names. */
void oracle_token_mixer(const double* z, int32_t T, int32_t D, int32_t dh, const float* w1, const float* b1,
                        const float* w3, const float* b3, const float* w2, const float* b2, const float* gain,
                        double eps, double* y) {
  double* mixed = (double*)malloc(sizeof(double) * (size_t)T * D * 3);
  double* f = mixed + (size_t)T * D;
  double* rv = f + (size_t)T * D;
  oracle_mix(z, T, D, mixed);
  for (int32_t j = 0; j < T; ++j) oracle_swiglu(mixed + j * D, D, dh, D, w1, b1, w3, b3, w2, b2, f + j * D);
  oracle_revert(f, T, D, rv);
  for (int32_t t = 0; t < T; ++t) {
    double res[1024];
    for (int32_t i = 0; i < D; ++i) res[i] = z[t * D + i] + rv[t * D + i];
    oracle_rmsnorm(res, D, gain, eps, y + t * D);
  }
  free(mixed);
}

/* PLE prediction layer (iQIYI CVR 3.2.4): single-layer fully connected experts e_k = ReLU(W_k y + b_k);
 * each task's gate is a softmax over all experts of (Wg_t y + bg_t); r_t = sum_k gate_t[k] e_k. */
void oracle_ple(const double* y, int32_t dy, int32_t n_experts, int32_t de, int32_t n_tasks, const float* const* we,
                const float* const* be, const float* const* wg, const float* const* bg, double* r, double* gates) {
  double* e = (double*)malloc(sizeof(double) * (size_t)n_experts * de);
  for (int32_t k = 0; k < n_experts; ++k) {
    linear(y, dy, de, we[k], be[k], e + (size_t)k * de);
    for (int32_t i = 0; i < de; ++i)
      if (e[(size_t)k * de + i] < 0.0) e[(size_t)k * de + i] = 0.0;
  }
  for (int32_t t = 0; t < n_tasks; ++t) {
    double g[ORACLE_MAX_EXPERTS];
    linear(y, dy, n_experts, wg[t], bg[t], g);
    double mx = g[0];
    for (int32_t k = 1; k < n_experts; ++k)
      if (g[k] > mx) mx = g[k];
    double sum = 0.0;
    for (int32_t k = 0; k < n_experts; ++k) {
      g[k] = exp(g[k] - mx);
      sum += g[k];
    }
    for (int32_t k = 0; k < n_experts; ++k) g[k] /= sum;
    if (gates)
      for (int32_t k = 0; k < n_experts; ++k) gates[t * n_experts + k] = g[k];
    for (int32_t i = 0; i < de; ++i) {
      double acc = 0.0;
      for (int32_t k = 0; k < n_experts; ++k) acc += g[k] * e[(size_t)k * de + i];
      r[(size_t)t * de + i] = acc;
    }
  }
  free(e);
}

/* Prediction head (iQIYI CVR 3.2.4): two fully connected layers with a non-linearity, read as
 * ReLU(W1 r + b1) then a single output, turned into pCVR by a sigmoid. */
double oracle_head(const double* r, int32_t de, int32_t dh, const float* w1, const float* b1, const float* w2,
                   const float* b2) {
  double h[1024];
  linear(r, de, dh, w1, b1, h);
  for (int32_t i = 0; i < dh; ++i)
    if (h[i] < 0.0) h[i] = 0.0;
  double logit;
  linear(h, dh, 1, w2, b2, &logit);
  return 1.0 / (1.0 + exp(-logit));
}

int32_t oracle_threads(int32_t threads) {
#ifdef _OPENMP
  return threads > 0 ? threads : omp_get_max_threads();
#else
  (void)threads;
  return 1;
#endif
}

/* ------------------------------------------------------------------------------------------ */
static int check_model(const oracle_model* m) {
  if (m->n_groups < 1 || m->n_groups > ORACLE_MAX_GROUPS || m->n_layers < 1 || m->n_layers > ORACLE_MAX_LAYERS ||
      m->n_experts < 1 || m->n_experts > ORACLE_MAX_EXPERTS || m->n_tasks < 1 || m->n_tasks > ORACLE_MAX_TASKS)
    return ORACLE_E_ARG;
  const int32_t T = m->n_tokens + m->n_groups;
  if (m->emb_dim > 512 || m->token_dim > 1024 || m->head_hidden > 1024 || m->token_dim % T != 0 ||
      m->token_dim % m->heads != 0 || m->seq_cols * m->emb_dim != m->token_dim)
    return ORACLE_E_ARG;
  return ORACLE_OK;
}

/* One request: its user bags, its sequences and every one of its candidates. */
/* lens[g]: events of group g that this request really has (the first lens[g] of its seq_len[g] slots);
 * the remaining slots are padding: never read, left out of the mean and masked out of the attention
 * (sequence lengths are a dynamic input, iQIYI CVR 3.3; sequences are padded, 3.4.2). A group with no
 * event decodes to a zero token and has a zero mean, as an empty bag pools to zero. */
static int score_request(const oracle_model* m, const oracle_table* tables, const oracle_weights* w, int32_t n_req,
                         int32_t r, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_offsets,
                         const int64_t* bag_ids, const int64_t* seq_ids, const int32_t* lens, double* out,
                         const oracle_dumps* dumps) {
  const int32_t Fu = m->n_user_fields, Fi = m->n_item_fields, E = m->emb_dim, D = m->token_dim;
  const int32_t N = m->n_tokens, G = m->n_groups, T = N + G;
  int32_t SL = 0;
  for (int32_t g = 0; g < G; ++g) SL += m->seq_len[g];
  int status = ORACLE_OK;

  /* user side: Fu mean-pooled bags -> clamp -> bf16 (one per request; iQIYI CVR 3.4.5) */
  double* u = (double*)malloc(sizeof(double) * (size_t)Fu * E);
  for (int32_t f = 0; f < Fu; ++f) {
    const int64_t bag = (int64_t)r * Fu + f;
    float pooled[512];
    int64_t* rows_out = dumps && dumps->rows ? dumps->rows + bag_offsets[bag] : NULL;
    int st = oracle_pool_bag(&tables[f], bag_ids + bag_offsets[bag], bag_offsets[bag + 1] - bag_offsets[bag], E,
                             m->clamp, pooled, rows_out);
    if (st) status = st;
    if (dumps && dumps->pooled) memcpy(dumps->pooled + bag * E, pooled, sizeof(float) * (size_t)E);
    for (int32_t c = 0; c < E; ++c) u[f * E + c] = oracle_bf16(pooled[c]);
  }

  /* sequences: each event concatenates seq_cols rows of the shared table (iQIYI CVR 3.2.1),
   * clamped and cast like the other lookups, then the group's SwiGLU (3.2.2) */
  double* H = (double*)malloc(sizeof(double) * (size_t)SL * D);
  const oracle_table* st_tab = &tables[Fu + Fi];
  int32_t base = 0;
  for (int32_t g = 0; g < G; ++g) {
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int32_t l = 0; l < lens[g]; ++l) {
      double x[1024];
      float row[512];
      const int64_t* ids = seq_ids + ((int64_t)r * SL + base + l) * m->seq_cols;
      for (int32_t c = 0; c < m->seq_cols; ++c) {
        int64_t id = ids[c];
        if (id < 0 || id >= st_tab->rows) {
          id = 0;
          bad = 1;
        }
        table_row(st_tab, id, E, row);
        for (int32_t k = 0; k < E; ++k) {
          float v = row[k];
          if (v > (float)m->clamp) v = (float)m->clamp;
          if (v < -(float)m->clamp) v = -(float)m->clamp;
          x[c * E + k] = oracle_bf16(v);
        }
      }
      oracle_swiglu(x, D, m->ffn_hidden, D, w->seq_w1[g], w->seq_b1[g], w->seq_w3[g], w->seq_b3[g], w->seq_w2[g],
                    w->seq_b2[g], H + (size_t)(base + l) * D);
    }
    if (bad) status = ORACLE_E_ID_RANGE;
    base += m->seq_len[g];
  }
  if (dumps && dumps->H) memcpy(dumps->H + (size_t)r * SL * D, H, sizeof(double) * (size_t)SL * D);

  /* mean-pooled sequence vector per group (iQIYI CVR 3.2.3, Query Decoding item 1), read as the
   * mean over positions of the encoded states */
  double* mg = (double*)calloc((size_t)G * D, sizeof(double));
  base = 0;
  for (int32_t g = 0; g < G; ++g) {
    for (int32_t i = 0; i < D; ++i) {
      double acc = 0.0;
      for (int32_t l = 0; l < lens[g]; ++l) acc += H[(size_t)(base + l) * D + i];
      mg[g * D + i] = lens[g] > 0 ? acc / lens[g] : 0.0;
    }
    base += m->seq_len[g];
  }

  /* candidates of this request */
  int bad_c = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad_c)
  for (int32_t b = 0; b < n_cand; ++b) {
    if (req_ids[b] != r) continue;
    double it[1024];
    for (int32_t f = 0; f < Fi; ++f) {
      const int64_t bag = (int64_t)n_req * Fu + (int64_t)b * Fi + f;
      float pooled[512];
      int64_t* rows_out = dumps && dumps->rows ? dumps->rows + bag_offsets[bag] : NULL;
      int st = oracle_pool_bag(&tables[Fu + f], bag_ids + bag_offsets[bag], bag_offsets[bag + 1] - bag_offsets[bag],
                               E, m->clamp, pooled, rows_out);
      if (st) bad_c = 1;
      if (dumps && dumps->pooled) memcpy(dumps->pooled + bag * E, pooled, sizeof(float) * (size_t)E);
      for (int32_t c = 0; c < E; ++c) it[f * E + c] = oracle_bf16(pooled[c]);
    }
    double* z = (double*)malloc(sizeof(double) * (size_t)T * D * 2);
    double* y = z + (size_t)T * D;
    oracle_tokenize(u, Fu * E, it, Fi * E, w->tok_w, w->tok_b, N, D, z); /* tokens x_1..x_N */
    for (int32_t layer = 0; layer < m->n_layers; ++layer) {
      if (layer > 0) memcpy(z, y, sizeof(double) * (size_t)N * D); /* stacked layer: x = previous Y[0:N] */
      int32_t gbase = 0;
      for (int32_t g = 0; g < G; ++g) {
        double q[1024];
        oracle_query(z, N, D, mg + g * D, w->q_w[layer][g], w->q_b[layer][g], q);
        if (dumps && dumps->Q) memcpy(dumps->Q + (((size_t)layer * n_cand + b) * G + g) * D, q, sizeof(double) * D);
        if (lens[g] > 0)
          oracle_cross_attention(q, H + (size_t)gbase * D, lens[g], D, m->heads, m->tau, z + (size_t)(N + g) * D,
                                 NULL);
        else
          for (int32_t i = 0; i < D; ++i) z[(size_t)(N + g) * D + i] = 0.0;
        gbase += m->seq_len[g];
      }
      if (dumps && dumps->Z)
        memcpy(dumps->Z + ((size_t)layer * n_cand + b) * T * D, z, sizeof(double) * (size_t)T * D);
      oracle_token_mixer(z, T, D, m->ffn_hidden, w->tm_w1[layer], w->tm_b1[layer], w->tm_w3[layer], w->tm_b3[layer],
                         w->tm_w2[layer], w->tm_b2[layer], w->tm_gain[layer], m->rms_eps, y);
      if (dumps && dumps->Y)
        memcpy(dumps->Y + ((size_t)layer * n_cand + b) * T * D, y, sizeof(double) * (size_t)T * D);
    }
    double rt[ORACLE_MAX_TASKS * 1024];
    oracle_ple(y, T * D, m->n_experts, m->expert_dim, m->n_tasks, w->ple_w, w->ple_b, w->gate_w, w->gate_b, rt, NULL);
    if (dumps && dumps->R)
      memcpy(dumps->R + (size_t)b * m->n_tasks * m->expert_dim, rt, sizeof(double) * (size_t)m->n_tasks * m->expert_dim);
    for (int32_t t = 0; t < m->n_tasks; ++t)
      out[(size_t)b * m->n_tasks + t] = oracle_head(rt + (size_t)t * m->expert_dim, m->expert_dim, m->head_hidden,
                                                    w->head_w1[t], w->head_b1[t], w->head_w2[t], w->head_b2[t]);
    free(z);
  }
  if (bad_c) status = ORACLE_E_ID_RANGE;
  free(mg);
  free(H);
  free(u);
  return status;
}

int oracle_score(const oracle_model* m, const oracle_table* tables, const oracle_weights* w, int32_t n_req,
                 int32_t n_cand, const int32_t* req_ids, const int64_t* bag_offsets, const int64_t* bag_ids,
                 const int64_t* seq_ids, const int32_t* req_subset, int32_t n_subset, double* out,
                 const oracle_dumps* dumps, int32_t threads) {
  return oracle_score_lens(m, tables, w, n_req, n_cand, req_ids, bag_offsets, bag_ids, seq_ids, NULL, req_subset,
                           n_subset, out, dumps, threads);
}

int oracle_score_lens(const oracle_model* m, const oracle_table* tables, const oracle_weights* w, int32_t n_req,
                      int32_t n_cand, const int32_t* req_ids, const int64_t* bag_offsets, const int64_t* bag_ids,
                      const int64_t* seq_ids, const int32_t* seq_lens, const int32_t* req_subset, int32_t n_subset,
                      double* out, const oracle_dumps* dumps, int32_t threads) {
  if (check_model(m) || n_req < 0 || n_cand < 0) return ORACLE_E_ARG;
  if (seq_lens)
    for (int64_t i = 0; i < (int64_t)n_req * m->n_groups; ++i)
      if (seq_lens[i] < 0 || seq_lens[i] > m->seq_len[i % m->n_groups]) return ORACLE_E_ARG;
#ifdef _OPENMP
  const int saved = omp_get_max_threads();
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  int status = ORACLE_OK;
  const int32_t n = req_subset ? n_subset : n_req;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t r = req_subset ? req_subset[i] : i;
    if (r < 0 || r >= n_req) {
      status = ORACLE_E_ARG;
      break;
    }
    const int32_t* lens = seq_lens ? seq_lens + (int64_t)r * m->n_groups : m->seq_len;
    int st = score_request(m, tables, w, n_req, r, n_cand, req_ids, bag_offsets, bag_ids, seq_ids, lens, out, dumps);
    if (st) status = st;
  }
#ifdef _OPENMP
  omp_set_num_threads(saved);
#endif
  return status;
}
