/* CPU oracle of the HyFormer-style CVR scoring forward pass -- TEST INFRASTRUCTURE.
 *
 * A plain, slow, loop-nest restatement of what the scoring path computes, in fp64,
 * written from the model description in the iQIYI ad-CVR article
 * ("爱奇艺广告CVR模型参数量10倍增长 ...", m.bobobaike.com/news/370088.html, sections
 * 3.1, 3.2.1-3.2.4 and 3.4.5) and the clamp / precision rules of the GPU CTR inference
 * article ("广告 CTR 预估模型的 GPU 推理优化", gtnt.cn/news/20674, section 三).
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * library. It shares no code with the CUDA path; both take their inputs from the seeded
 * generator in synth/.
 *
 * Precision: the exact parts are the pooled embedding means (fp32 sum in bag order from
 * 0.0f, one IEEE division, clamp) and the casts to bf16 that the method itself specifies
 * (pooled embeddings and sequence rows are cast to half precision after the lookup; the
 * dense weights are bf16 values). Everything after those casts is fp64.
 */
#ifndef CVR_ORACLE_H
#define CVR_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_MAX_GROUPS 3
#define ORACLE_MAX_LAYERS 4
#define ORACLE_MAX_EXPERTS 8
#define ORACLE_MAX_TASKS 4

typedef struct {
  int32_t n_user_fields, n_item_fields, emb_dim, n_tokens, token_dim, n_groups;
  int32_t seq_len[ORACLE_MAX_GROUPS];
  int32_t seq_cols, ffn_hidden, heads, n_layers, n_experts, expert_dim, n_tasks, head_hidden;
  double tau, clamp, rms_eps;
} oracle_model;

/* One embedding table: materialised (data != NULL, [rows][emb_dim] fp32) or evaluated on
 * demand from the seeded generator (data == NULL: seed, index, scale). */
typedef struct {
  const float* data;
  int64_t rows;
  uint64_t seed;
  uint32_t index;
  double scale;
} oracle_table;

/* Dense weights, fp32 arrays holding bf16 values, [out][in] row-major. */
typedef struct {
  const float *tok_w, *tok_b;
  const float *seq_w1[ORACLE_MAX_GROUPS], *seq_b1[ORACLE_MAX_GROUPS], *seq_w3[ORACLE_MAX_GROUPS],
      *seq_b3[ORACLE_MAX_GROUPS], *seq_w2[ORACLE_MAX_GROUPS], *seq_b2[ORACLE_MAX_GROUPS];
  const float *q_w[ORACLE_MAX_LAYERS][ORACLE_MAX_GROUPS], *q_b[ORACLE_MAX_LAYERS][ORACLE_MAX_GROUPS];
  const float *tm_w1[ORACLE_MAX_LAYERS], *tm_b1[ORACLE_MAX_LAYERS], *tm_w3[ORACLE_MAX_LAYERS],
      *tm_b3[ORACLE_MAX_LAYERS], *tm_w2[ORACLE_MAX_LAYERS], *tm_b2[ORACLE_MAX_LAYERS], *tm_gain[ORACLE_MAX_LAYERS];
  const float *ple_w[ORACLE_MAX_EXPERTS], *ple_b[ORACLE_MAX_EXPERTS];
  const float *gate_w[ORACLE_MAX_TASKS], *gate_b[ORACLE_MAX_TASKS];
  const float *head_w1[ORACLE_MAX_TASKS], *head_b1[ORACLE_MAX_TASKS], *head_w2[ORACLE_MAX_TASKS],
      *head_b2[ORACLE_MAX_TASKS];
} oracle_weights;

/* Optional intermediate outputs (any pointer may be NULL). Only the requests that are
 * scored are written. */
typedef struct {
  float* pooled;   /* [n_req*Fu + n_cand*Fi][emb_dim]: clamped fp32 means, in bag order */
  int64_t* rows;   /* [nnz]: row actually read for each id (the id, or 0 when out of range) */
  double* H;       /* [n_req][sum_len][token_dim]: encoded sequence states */
  double* Q;       /* [n_layers][n_cand][n_groups][token_dim]: queries */
  double* Z;       /* [n_layers][n_cand][n_tokens+n_groups][token_dim]: token-mixer inputs */
  double* Y;       /* [n_layers][n_cand][n_tokens+n_groups][token_dim]: token-mixer outputs */
  double* R;       /* [n_cand][n_tasks][expert_dim]: gated expert mixtures */
} oracle_dumps;

/* Status codes */
#define ORACLE_OK 0
#define ORACLE_E_ARG 1
#define ORACLE_E_ID_RANGE 3

/* Scores the candidates of the requests in req_subset[0..n_subset) (all requests when
 * req_subset == NULL), writing out[b][task] = pCVR for each of their candidates b.
 * tables: [n_user_fields + n_item_fields + 1], the last one the shared sequence table.
 * threads <= 0 uses the OpenMP default. Returns ORACLE_E_ID_RANGE when an id is out of range
 * (the row read is then row 0), ORACLE_E_ARG on bad sizes. */
int oracle_score(const oracle_model* m, const oracle_table* tables, const oracle_weights* w, int32_t n_req,
                 int32_t n_cand, const int32_t* req_ids, const int64_t* bag_offsets, const int64_t* bag_ids,
                 const int64_t* seq_ids, const int32_t* req_subset, int32_t n_subset, double* out,
                 const oracle_dumps* dumps, int32_t threads);

/* As oracle_score with variable-length sequences: seq_lens[n_req][n_groups] gives the events each request
 * really has in each group, 0 <= seq_lens <= seq_len[g] (else ORACLE_E_ARG); the slots past it are padding,
 * never read, out of the mean and masked out of the attention; a group with no event decodes to zero. */
int oracle_score_lens(const oracle_model* m, const oracle_table* tables, const oracle_weights* w, int32_t n_req,
                      int32_t n_cand, const int32_t* req_ids, const int64_t* bag_offsets, const int64_t* bag_ids,
                      const int64_t* seq_ids, const int32_t* seq_lens, const int32_t* req_subset, int32_t n_subset,
                      double* out, const oracle_dumps* dumps, int32_t threads);

/* ---- single stages, exposed so that each can be pinned on its own ---- */
int oracle_pool_bag(const oracle_table* t, const int64_t* ids, int64_t n, int32_t dim, double clamp, float* out,
                    int64_t* rows_out);
double oracle_bf16(float x);
void oracle_swiglu(const double* x, int32_t din, int32_t dh, int32_t dout, const float* w1, const float* b1,
                   const float* w3, const float* b3, const float* w2, const float* b2, double* y);
void oracle_tokenize(const double* u, int32_t du, const double* it, int32_t di, const float* w, const float* b,
                     int32_t n_tokens, int32_t token_dim, double* x);
void oracle_query(const double* x, int32_t n_tokens, int32_t token_dim, const double* m_g, const float* w,
                  const float* b, double* q);
void oracle_cross_attention(const double* q, const double* H, int32_t L, int32_t token_dim, int32_t heads,
                            double tau, double* d, double* probs /* [heads][L] or NULL */);
void oracle_mix(const double* z, int32_t T, int32_t D, double* mixed);
void oracle_revert(const double* mixed, int32_t T, int32_t D, double* z);
void oracle_rmsnorm(const double* x, int32_t D, const float* gain, double eps, double* y);
void oracle_token_mixer(const double* z, int32_t T, int32_t D, int32_t dh, const float* w1, const float* b1,
                        const float* w3, const float* b3, const float* w2, const float* b2, const float* gain,
                        double eps, double* y);
void oracle_ple(const double* y, int32_t dy, int32_t n_experts, int32_t de, int32_t n_tasks,
                const float* const* we, const float* const* be, const float* const* wg, const float* const* bg,
                double* r /* [n_tasks][de] */, double* gates /* [n_tasks][n_experts] or NULL */);
double oracle_head(const double* r, int32_t de, int32_t dh, const float* w1, const float* b1, const float* w2,
                   const float* b2);
int32_t oracle_threads(int32_t threads);

#ifdef __cplusplus
}
#endif
#endif
