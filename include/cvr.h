/*
 * cvr.h -- C ABI of the GB300 CVR scoring library.
 *
 * The library scores ad candidates with the HyFormer-style CVR ranking model described in the
 * iQIYI ad-CVR article ("爱奇艺广告CVR模型参数量10倍增长 ...", m.bobobaike.com/news/370088.html):
 *
 *   1. mean-pooled multi-hot embedding bags over fp32 tables (section 3.1 item 2; 3.2.1), clamped to
 *      [-clamp, clamp] and cast to bf16 after the lookup (GPU CTR inference article,
 *      gtnt.cn/news/20674, section 三);
 *   2. tokenisation of the non-sequence embedding [user ; item] into 13 tokens of 128 (3.2.2);
 *   3. a SwiGLU encoder per behaviour-sequence group, the three groups sharing one id table (3.2.1-3.2.2);
 *   4. Query Decoding: per group, one query from the 13 tokens and the mean-pooled encoded sequence,
 *      cross-attending over that sequence with a temperature-scaled softmax (3.2.3);
 *   5. the Query Boosting Token Mixer over 16 tokens: split -> mix -> SwiGLU -> revert, residual,
 *      RMSNorm (3.2.3); steps 4-5 stack n_layers times;
 *   6. a PLE of 3 single-layer experts with per-task softmax gates and a two-layer head per task,
 *      ending in a sigmoid pCVR (3.2.4).
 *
 * Requests follow the user/item split of section 3.4.5: each request carries one user (user bags,
 * behaviour sequences) and many candidates (item bags), linked by a per-candidate request id; all
 * user-side work runs once per request. Every per-call size is an argument (section 3.3).
 *
 * All work runs in hand-written sm_103a CUDA kernels on the device and stream given at creation.
 * Conventions:
 *  - Per-call pointers of cvr_score are DEVICE pointers, borrowed for the duration of the call.
 *  - Calls are synchronous: they return after the batch is scored and the device error word read.
 *  - No call aborts, traps or waits on a device flag without a time limit.
 *  - A handle is not thread-safe; use one handle per host thread / stream.
 */
#ifndef CVR_H
#define CVR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CVR_MAX_LAYERS 4
#define CVR_N_USER_FIELDS 8
#define CVR_N_ITEM_FIELDS 8
#define CVR_N_GROUPS 3
#define CVR_N_EXPERTS 3
#define CVR_N_TASKS 2

typedef enum {
  CVR_OK = 0,
  CVR_E_ARG = 1,      /* null pointer, unsupported configuration or option */
  CVR_E_SHAPE = 2,    /* a size out of range */
  CVR_E_ID_RANGE = 3, /* an id outside its table; the id read row 0 and `out` is not meaningful */
  CVR_E_OOM = 4,      /* device or pinned-host allocation failed */
  CVR_E_CUDA = 5,     /* a CUDA call failed (message in cvr_last_error) */
  CVR_E_INPUT = 6,    /* bag offsets decreasing, or request ids out of range / decreasing */
  CVR_E_TIMEOUT = 7   /* a bounded device-side wait gave up (reported instead of hanging) */
} cvr_status;

typedef struct cvr_handle cvr_handle;

/* Model configuration. The kernels are built for the dimensions of the model above; the fixed
 * fields must hold exactly the values in brackets, otherwise cvr_create returns CVR_E_ARG. */
typedef struct {
  int32_t n_user_fields; /* [8]  user/context fields, one bag each per request */
  int32_t n_item_fields; /* [8]  item fields, one bag each per candidate */
  int32_t emb_dim;       /* [32] embedding width of every table */
  int32_t n_tokens;      /* [13] non-sequence tokens N */
  int32_t token_dim;     /* [128] */
  int32_t n_groups;      /* [3]  behaviour-sequence groups */
  int32_t seq_len[3];    /* events per request in each group, >= 1 */
  int32_t seq_cols;      /* [4]  id columns per event (rows of the shared table, concatenated) */
  int32_t ffn_hidden;    /* [256] SwiGLU hidden width (sequence encoder and Token Mixer) */
  int32_t heads;         /* [4]  cross-attention heads (of token_dim / heads = 32) */
  int32_t n_layers;      /* 1 .. CVR_MAX_LAYERS stacked Query Decoding + Token Mixer layers */
  int32_t n_experts;     /* [3]  PLE experts */
  int32_t expert_dim;    /* [256] */
  int32_t n_tasks;       /* [2]  tasks, one pCVR each */
  int32_t head_hidden;   /* [128] */
  float tau;             /* softmax temperature: logits are q.k / (tau * sqrt(32)), > 0 */
  float clamp;           /* embeddings are clamped to [-clamp, clamp] after pooling / lookup, > 0 */
  float rms_eps;         /* RMSNorm epsilon, >= 0 */
  int64_t user_rows[8];  /* rows of each user-field table, >= 1 */
  int64_t item_rows[8];  /* rows of each item-field table, >= 1 */
  int64_t seq_rows;      /* rows of the shared sequence table, >= 1 */
} cvr_config;

/* Weights. Tables are DEVICE fp32 [rows][32] arrays, BORROWED: they must stay valid and unchanged
 * for the life of the handle. Dense weights are HOST fp32 arrays in [out][in] row-major layout
 * (biases [out]); they are COPIED and rounded to bf16 (round-to-nearest-even) at creation, except the
 * biases, RMSNorm gains and the last head layer, which stay fp32. Every pointer is required. */
typedef struct {
  const float* user_tables[8];
  const float* item_tables[8];
  const float* seq_table;
  const float* tok_w; /* [13*128][512]: [user 256 ; item 256] -> 13 tokens of 128 */
  const float* tok_b; /* [1664] */
  const float *seq_w1[3], *seq_b1[3]; /* [256][128], [256]   group encoders: */
  const float *seq_w3[3], *seq_b3[3]; /* [256][128], [256]   W2(silu(W1 x+b1)*(W3 x+b3))+b2 */
  const float *seq_w2[3], *seq_b2[3]; /* [128][256], [128] */
  const float *q_w[CVR_MAX_LAYERS][3], *q_b[CVR_MAX_LAYERS][3]; /* [128][13*128+128], [128] query FFN */
  const float *tm_w1[CVR_MAX_LAYERS], *tm_b1[CVR_MAX_LAYERS];   /* [256][128], [256] Token Mixer SwiGLU */
  const float *tm_w3[CVR_MAX_LAYERS], *tm_b3[CVR_MAX_LAYERS];   /* [256][128], [256] */
  const float *tm_w2[CVR_MAX_LAYERS], *tm_b2[CVR_MAX_LAYERS];   /* [128][256], [128] */
  const float* tm_gain[CVR_MAX_LAYERS];                          /* [128] RMSNorm gain */
  const float *ple_w[3], *ple_b[3];     /* [256][2048], [256] experts over the 16 x 128 tokens */
  const float *gate_w[2], *gate_b[2];   /* [3][2048], [3]     per-task gates */
  const float *head_w1[2], *head_b1[2]; /* [128][256], [128] */
  const float *head_w2[2], *head_b2[2]; /* [1][128], [1] */
} cvr_weights;

/* Creates a scorer on the current CUDA device, working on `cuda_stream` (a cudaStream_t; NULL =
 * the legacy default stream). Returns CVR_E_ARG for a bad configuration or a null weight pointer,
 * CVR_E_OOM / CVR_E_CUDA on device failures. On success *out owns device memory until cvr_destroy. */
cvr_status cvr_create(const cvr_weights* weights, const cvr_config* cfg, void* cuda_stream, cvr_handle** out);

/* Scores one batch of n_req requests and n_cand candidates (all DEVICE pointers):
 *   req_ids     [n_cand] int32: request index of each candidate, in [0, n_req), non-decreasing.
 *   bag_offsets [n_req*8 + n_cand*8 + 1] int64 CSR offsets into bag_ids: first the user bags in
 *               (request, field) order, then the item bags in (candidate, field) order; non-negative and
 *               non-decreasing (normally bag_offsets[0] = 0). A negative or decreasing offset returns
 *               CVR_E_INPUT and its bag is read as empty.
 *   bag_ids     [bag_offsets[last]] int64 row ids, local to each field's table. An empty bag pools to 0.
 *   seq_ids     [n_req][sum(seq_len)][4] int64 rows of the shared sequence table; per request the
 *               events of group 0, then group 1, then group 2.
 *   out         [n_cand][2] fp32 pCVR per task, written by the call (caller-owned).
 * Sizes: 1 <= n_req <= 65535, 1 <= n_cand <= 2^20. Workspace grows on demand (first call at a size allocates).
 * Returns CVR_E_SHAPE on sizes out of range, CVR_E_ID_RANGE / CVR_E_INPUT on bad ids, offsets or
 * request ids (detected on the device, never read out of bounds), CVR_E_CUDA on CUDA errors.
 * When the sequence encoder leaves SMs free, part of a call runs on a second stream owned by the handle; it
 * forks from the handle's stream after the call's first kernel and joins it again before the attention, so
 * a call stays ordered on the handle's stream like one sequence of kernels. */
cvr_status cvr_score(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_ids,
                     const int64_t* bag_offsets, const int64_t* seq_ids, float* out);

/* As cvr_score, but only enqueues the work on the handle's stream and returns CVR_OK (or a host-side
 * error: CVR_E_ARG / CVR_E_SHAPE / CVR_E_OOM / CVR_E_CUDA) without waiting. The input and output buffers
 * must stay valid until cvr_sync returns. Several calls may be in flight; their device-side error bits
 * accumulate until the next cvr_sync. */
cvr_status cvr_score_async(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                           const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids, float* out);

/* As cvr_score with variable-length sequences (sequence lengths are a dynamic input, iQIYI ad-CVR article
 * 3.3; sequences are padded, 3.4.2): seq_lens [n_req][3] int32 (DEVICE) gives the events each request
 * really has in each group, 0 <= seq_lens[r][g] <= seq_len[g]; seq_ids keeps its padded layout and the
 * slots past a request's length are padding -- never read (any value is accepted there), left out of the
 * mean-pooled sequence vector and masked out of the cross-attention. A group with no event decodes to a
 * zero token and has a zero mean. A length outside the range returns CVR_E_INPUT (it is used clamped, so
 * nothing is read out of bounds). */
cvr_status cvr_score_varlen(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                            const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids,
                            const int32_t* seq_lens, float* out);
/* cvr_score_varlen, enqueued only (as cvr_score_async; collect the status with cvr_sync). */
cvr_status cvr_score_varlen_async(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                                  const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids,
                                  const int32_t* seq_lens, float* out);

/* Waits for every call enqueued on the handle's stream and returns the status of the device-side checks
 * of all calls since the previous cvr_sync (CVR_E_ID_RANGE, CVR_E_INPUT, CVR_E_TIMEOUT) or CVR_E_CUDA. */
cvr_status cvr_sync(cvr_handle* h);

/* As cvr_score, and also writes the exact pooled embeddings and the rows read (DEVICE pointers, each
 * may be NULL): pooled_fp32 [n_req*8 + n_cand*8][32] -- the clamped fp32 means of every bag, in
 * bag_offsets order, before the bf16 cast; rows [bag_offsets[last]] -- the row each id read (the id
 * itself, or 0 when out of range). */
cvr_status cvr_score_debug(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                           const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids, float* out,
                           float* pooled_fp32, int64_t* rows);

/* As cvr_score with HOST inputs and output (iQIYI ad-CVR article 3.4.1: input movement per batch).
 * An array in pinned, device-mapped host memory (cudaHostAlloc / cudaHostRegister; PyTorch's
 * pin_memory) or in managed memory is read -- `out` written -- in place by the kernels: on a
 * Grace-Blackwell node over NVLink-C2C, with no staging copy. Any other host array is copied to a
 * device staging buffer owned by the handle (one asynchronous copy per array), and `out` back. The call
 * waits for the stream once and returns the call's status. n_bag_ids = bag_offsets[last] (the length
 * of bag_ids). The caller must not modify the arrays until the call returns. */
cvr_status cvr_score_host(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_ids,
                          int64_t n_bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids, float* out);

/* Intermediate results of the last call, copied to `dst` (DEVICE) for inspection; `bytes` must equal
 * the stage's size for the last call, else CVR_E_SHAPE:
 *   CVR_STAGE_H   bf16 [group][request][position][128]: encoded sequence states
 *   CVR_STAGE_Z   bf16 [n_cand][16][128]: input of the last Token Mixer (13 tokens + 3 decoded tokens)
 *   CVR_STAGE_Q   bf16 [n_cand][3][128]: queries of the last layer
 *   CVR_STAGE_Y   bf16 [n_cand][16][128]: output of the last Token Mixer
 *   CVR_STAGE_EXPERTS bf16 [n_cand][768]: PLE expert outputs (after ReLU)
 *   CVR_STAGE_GATES fp32 [n_cand][8]: task gates (2 x 3, padded to 8)
 * The last two are written only by calls made with CVR_OPT_KEEP_STAGES set (else CVR_E_ARG). */
enum { CVR_STAGE_H = 0, CVR_STAGE_Z = 1, CVR_STAGE_Q = 2, CVR_STAGE_Y = 3, CVR_STAGE_EXPERTS = 4, CVR_STAGE_GATES = 5 };
cvr_status cvr_debug_stage(cvr_handle* h, int32_t stage, void* dst, int64_t bytes);

/* Options (cvr_set_option):
 *   CVR_OPT_ATTENTION_TC 1 = cross-attention on the tcgen05 kernel (S and O accumulated in tensor memory, one
 *                            CTA per 128 candidates and group); 0 = on the register-tile kernel (default 0:
 *                            with heads 32 wide its many small MMAs keep up better; both meet the same
 *                            tolerance)
 *   CVR_OPT_PROFILE      1 = record a CUDA event after every kernel of a call (read with cvr_stage_times);
 *                            such calls keep every kernel on the handle's stream, so each time is one kernel's
 *   CVR_OPT_CUDA_GRAPH   1 = replay the call's kernel sequence from a CUDA graph captured per (n_req, n_cand)
 *                            (default 1); 0 = launch eagerly
 *   CVR_OPT_PDL          1 = launch each kernel with programmatic dependent launch, so its prologue overlaps
 *                            the previous kernel (default 1); 0 = plain stream order
 *   CVR_OPT_PLE_INT8     1 = the PLE expert and gate GEMM reads its weights as 8-bit integers with one fp32 scale
 *                            per output row (scale = max|w| / 127, q = round-half-even(w / scale), made from the
 *                            fp32 weights at creation); activations stay bf16 and the scale is applied to the
 *                            fp32 sums, so the integers enter the tensor cores exactly. Outputs stay inside the
 *                            pCVR tolerance of the fp64 model on the production and two-layer workloads but
 *                            differ from the bf16 weights' (default 0: bf16 weights). Mixed-precision inference,
 *                            iQIYI ad-CVR article, outlook section.
 *   CVR_OPT_KEEP_STAGES  1 = calls also write the PLE expert outputs and gates, for CVR_STAGE_EXPERTS and
 *                            CVR_STAGE_GATES (default 0: not written; they are not needed for the scores) */
enum {
  CVR_OPT_PROFILE = 0,
  CVR_OPT_CUDA_GRAPH = 1,
  CVR_OPT_PDL = 2,
  CVR_OPT_ATTENTION_TC = 3,
  CVR_OPT_PLE_INT8 = 4,
  CVR_OPT_KEEP_STAGES = 5
};
cvr_status cvr_set_option(cvr_handle* h, int32_t option, int64_t value);

/* With CVR_OPT_PROFILE set: per-kernel device times of the last call, in launch order. Writes up to
 * `cap` entries of ms[] and names[] (static strings) and returns the count through *n. */
cvr_status cvr_stage_times(cvr_handle* h, float* ms, const char** names, int32_t cap, int32_t* n);

/* Number of kernels the last call launched (graph replays count the kernels in the graph). */
int32_t cvr_last_launch_count(const cvr_handle* h);

/* Human-readable detail of the last failure of this handle ("" if none). */
const char* cvr_last_error(const cvr_handle* h);
const char* cvr_status_string(cvr_status s);

/* Diagnostic (the pages have no counterpart): the per-CTA timeline of the forward-pass kernels, in builds compiled with
 * -DCVR_TIMELINE (otherwise CVR_E_ARG). The first thread of every CTA records the device clock (%globaltimer, ns) at
 * entry, when its wait for the previous kernel's data returned, and at exit: records [10 kernels][8192 CTAs][3]
 * (HOST uint64; 0 = not recorded; kernels in the order sparse, seq_mlp, seq_colsum, tokenizer, query, attention,
 * token_mixer, ple_heads, attention_tc; CTA = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z), CTAs
 * past 8192 not recorded; a stacked layer's launch overwrites the previous layer's). Waits for the handle's stream,
 * copies out when records is not NULL (n_records must be 245760), then clears every record when clear != 0. */
#define CVR_TIMELINE_RECORDS (10 * 8192 * 3)
cvr_status cvr_timeline(cvr_handle* h, uint64_t* records, int64_t n_records, int32_t clear);

/* Diagnostic (the pages have no counterpart): launches one CTA that waits on a barrier nothing arrives at,
 * through the same bounded wait as the scoring kernels, and returns what a call would report when a wait
 * gives up: CVR_E_TIMEOUT after about 1 s, the handle staying usable. Shows that a stuck wait ends as a
 * status instead of a hung GPU. */
cvr_status cvr_selftest_wait_timeout(cvr_handle* h);

/* The prediction step alone -- PLE experts and gates, task towers and sigmoid (one kernel) -- on a caller's Token Mixer
 * output, without allocating device memory. The papers have no counterpart: it serves callers that
 * cannot allocate mid-flight (a serving loop whose device memory is all pre-reserved by its own pool, or
 * one that cannot afford the device-wide synchronisation of cudaMalloc / cudaFree that a growing
 * cvr_score workspace would cost). Its intermediates live in one fixed device array of
 * CVR_NOALLOC_MAX_CAND x 1,024 + 512 bytes (1 MB) inside this library: the gate-weighted expert sums of every
 * candidate and the error word (the expert outputs and gates are not kept, whatever CVR_OPT_KEEP_STAGES says).
 *   y    DEVICE bf16 [n_cand][16][128]: the last Token Mixer's output (the layout of CVR_STAGE_Y), 16-byte
 *        aligned; read only.
 *   out  DEVICE fp32 [n_cand][2]: pCVR per task, written by the call (caller-owned).
 * 0 <= n_cand <= CVR_NOALLOC_MAX_CAND (0 does nothing); larger batches return CVR_E_SHAPE. Runs on the
 * handle's stream and waits for it, returning CVR_E_TIMEOUT / CVR_E_CUDA like cvr_score.
 * The first call on a device looks up the array's address (setup: make it before any stream capture).
 * The array is shared by every handle of the process on that device: calls whose execution overlaps
 * (on two streams, two handles or two threads) race on it. */
#define CVR_NOALLOC_MAX_CAND 1024
cvr_status cvr_predict_noalloc(cvr_handle* h, int32_t n_cand, const void* y, float* out);

/* Hot-row cache in HBM in front of one embedding table (GPU CTR inference article, section 二: the hot
 * rows live in GPU memory, a lookup tries them first and falls back to host DRAM). Meant for tables kept
 * in host memory that the GPU reads directly (pinned with cudaHostAlloc / cudaHostRegister; on a
 * Grace-Blackwell node over NVLink-C2C): pass such a table's address in cvr_weights like any other.
 *   table  0..7 user fields, 8..15 item fields, 16 the shared sequence table
 *   slots  a power of two in [1024, 2^28] (rows held; 128 + 16 bytes of HBM each), or 0 to remove it
 * Direct-mapped: slot = (id * 0x9E3779B97F4A7C15) >> (64 - log2(slots)). During a call the cache is only
 * read; a row that misses is read from the table and logged (up to 2^20 per call), and after the call a
 * logged row replaces its slot's row unless that row was read in the same call, so a hot row is never
 * pushed out by the cold rows of the call that used it. Cached rows are exact fp32 copies: results do not
 * depend on hits or misses. The tables must not change while a cache holds their rows. The handle's
 * captured graphs are dropped (the next call of each shape captures again); the call waits for the stream.
 * Errors: CVR_E_ARG (table or slots out of range), CVR_E_OOM. */
cvr_status cvr_cache_enable(cvr_handle* h, int32_t table, int64_t slots);

/* Cache lookups since the last read (all tables): rows served from a cache slot and rows read from their
 * table. Waits for the stream, then resets both counts. Both are 0 while no cache is enabled. */
cvr_status cvr_cache_stats(cvr_handle* h, int64_t* hits, int64_t* misses);

/* Frees the handle's device memory, graphs and events. NULL is ignored. */
void cvr_destroy(cvr_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* CVR_H */
