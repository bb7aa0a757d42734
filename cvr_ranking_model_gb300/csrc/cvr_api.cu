// Host side of the CVR scoring library: the C ABI of include/cvr.h.
//
// cvr_create packs the dense weights into the layouts the kernels consume (bf16, W1/W3 rows interleaved
// per 128 hidden units, the three query FFNs stacked, the PLE gates appended to the expert rows) and
// builds their TMA tensor maps. cvr_score validates sizes on the host, grows the workspace for the
// batch if needed, and runs the forward pass -- eagerly or by replaying a CUDA graph captured for the
// batch's (n_req, n_cand) bucket (iQIYI ad-CVR article 3.4.4) -- then reads the device error word.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/cvr.h"
#include "cvr_internal.cuh"

using namespace cvr;
typedef __nv_bfloat16 bf16;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

uint16_t f32_to_bf16_bits(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

float bf16_round(float x) {
  const uint32_t u = (uint32_t)f32_to_bf16_bits(x) << 16;
  float r;
  std::memcpy(&r, &u, 4);
  return r;
}

struct GraphEntry {
  cudaGraphExec_t exec = nullptr;
  std::vector<const void*> key;
  int launches = 0;
};

const char* kStageNames[] = {"sparse", "seq_mlp", "seq_colsum", "tokenizer", "query", "attention", "token_mixer",
                             "ple_heads", "cache_admit"};

}  // namespace

struct cvr_handle {
  int device = 0;
  int num_sms = 1;
  cudaStream_t stream = nullptr;
  cudaStream_t cap_stream = nullptr;
  // the tokeniser's token columns run on a second stream, next to the sequence encoder (fork after the
  // sparse kernel, join before the query columns)
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_tail = nullptr;
  cvr_config cfg{};
  int n_layers = 1, SL = 0;
  int L[kG] = {0, 0, 0};
  std::string last_error;
  // packed weights
  void* wblob = nullptr;
  size_t wblob_bytes = 0;
  void* w8blob = nullptr;    // PLE expert and gate rows as int8 [4 x 208][2048], then their fp32 scales [4 x 208]
  float* ple_s8 = nullptr;
  bool ple_int8 = false;     // the PLE runs on the 8-bit rows
  bf16 *tokI = nullptr, *tokU = nullptr, *seqW13 = nullptr, *seqW2 = nullptr, *qX = nullptr, *qm = nullptr;
  bf16 *tmW13 = nullptr, *tmW2 = nullptr, *pleW = nullptr, *headW1 = nullptr;
  float *tok_b = nullptr, *seq_b13 = nullptr, *seq_b2 = nullptr, *q_b = nullptr, *tm_b13 = nullptr, *tm_b2 = nullptr;
  float *tm_gain = nullptr, *ple_b = nullptr, *head_b1 = nullptr, *head_w2 = nullptr, *head_b2 = nullptr;
  const float* tables[kFu + kFi + 1] = {};
  int64_t rows[kFu + kFi + 1] = {};
  // workspace
  int R_cap = 0, B_cap = 0, max_chunks = 0;
  void* ws = nullptr;
  bf16 *U = nullptr, *I = nullptr, *Xs = nullptr, *H = nullptr, *Z = nullptr, *Y = nullptr, *Q = nullptr, *Ex = nullptr;
  float *colsum = nullptr, *xu = nullptr, *qb = nullptr, *gates = nullptr;
  int* err = nullptr;
  unsigned* cs_count = nullptr;
  unsigned* ple_ready = nullptr;  // per 128-row block: Token Mixer tiles written
  unsigned* attn_ready = nullptr;  // per 32-candidate block: attention groups written (same allocation)
  bf16* Rt = nullptr;             // [2][B_cap][256] gate-weighted expert sums
  unsigned* xu_ready = nullptr;   // [R_cap/128][16] user row-tiles of the tokeniser written
  int32_t* req_copy = nullptr;  // the call's request ids in the workspace
  float* attn_state = nullptr;
  unsigned* attn_count = nullptr;
  int attn_splits = 1;
  int* err_host = nullptr;      // pinned, mapped: the call's error bits
  int* err_host_dev = nullptr;  // its device address
  // host-input staging
  void* stage = nullptr;
  size_t stage_bytes = 0;
  // tensor maps
  CUtensorMap tm_seqW13, tm_seqW2, tm_tokI, tm_tokU, tm_qW[kMaxLayers], tm_qWw[kMaxLayers], tm_tmW13, tm_tmW2, tm_pleW, tm_pleW8, tm_headW1;
  CUtensorMap tm_Xs, tm_I, tm_U, tm_U32, tm_x_Z, tm_x_Y, tm_full_Z, tm_full_Y, tm_Q, tm_H, tm_R, tm_Ex;
  // graphs, profiling
  bool use_graph = true, profile = false, pdl = true;
  bool keep_stages = false;  // the PLE also writes the expert outputs and gates (for cvr_debug_stage)
  bool last_kept = false;    // ... and the last call did
  bool attn_tc = false;  // cross-attention on the tcgen05 kernel instead of the register-tile one
  bool last_q_add = false;  // the last call left the first layer's queries without their mean-pooled term
  // hot-row caches in HBM, per table (slots == 0: none)
  int64_t c_slots[kNTab] = {};
  float* c_rows[kNTab] = {};
  int64_t* c_tags[kNTab] = {};
  unsigned* c_use[kNTab] = {};
  unsigned* c_claim[kNTab] = {};
  int64_t* miss_list = nullptr;
  unsigned* cache_ctl = nullptr;             // misses logged, epoch, admission block counter
  unsigned long long* cache_stat = nullptr;  // hits, misses
  std::map<std::pair<int, int>, GraphEntry> graphs;
  std::vector<cudaEvent_t> events;
  std::vector<const char*> event_names;
  int n_events_last = 0;
  int last_launches = 0;
  int last_R = 0, last_B = 0;
  bf16 *last_zin = nullptr, *last_zout = nullptr;
};

namespace {

cvr_status fail(cvr_handle* h, cvr_status s, const std::string& msg) {
  if (h) h->last_error = msg;
  return s;
}
cvr_status cuda_fail(cvr_handle* h, cudaError_t e, const char* what) {
  return fail(h, CVR_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
               uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit rows [outer][inner] bytes (row stride `row_stride` bytes), unswizzled boxes of box_inner x box_outer
bool encode_2d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride,
                  uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cvr_status check_config(const cvr_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return CVR_E_ARG;
  };
  if (c->n_user_fields != kFu || c->n_item_fields != kFi || c->emb_dim != kE || c->n_tokens != kN ||
      c->token_dim != kD || c->n_groups != kG || c->seq_cols != kCols || c->ffn_hidden != kHid ||
      c->heads != kHeads || c->n_experts != kNE || c->expert_dim != kDE || c->n_tasks != kNT ||
      c->head_hidden != kHH)
    return bad("unsupported model dimensions (the kernels are built for 8+8 fields of 32, 13 tokens of 128, "
               "3 groups x 4 columns, SwiGLU 256, 4 heads, 3 experts of 256, 2 tasks, head 128)");
  if (c->n_layers < 1 || c->n_layers > CVR_MAX_LAYERS) return bad("n_layers must be in [1, 4]");
  for (int g = 0; g < kG; ++g)
    if (c->seq_len[g] < 1 || c->seq_len[g] > (1 << 20)) return bad("seq_len must be in [1, 2^20]");
  if (!(c->tau > 0.f) || !(c->clamp > 0.f) || !(c->rms_eps >= 0.f) || !std::isfinite(c->tau) ||
      !std::isfinite(c->clamp) || !std::isfinite(c->rms_eps))
    return bad("tau and clamp must be positive and finite, rms_eps finite and >= 0");
  for (int f = 0; f < kFu; ++f)
    if (c->user_rows[f] < 1) return bad("user_rows must be >= 1");
  for (int f = 0; f < kFi; ++f)
    if (c->item_rows[f] < 1) return bad("item_rows must be >= 1");
  if (c->seq_rows < 1) return bad("seq_rows must be >= 1");
  return CVR_OK;
}

// ---- weight packing ----
struct Packer {
  std::vector<uint16_t> bf;   // bf16 blob
  std::vector<float> f32;     // fp32 blob
  size_t add_bf(size_t n) {
    size_t off = bf.size();
    bf.resize(off + ((n + 63) / 64) * 64, 0);  // 128-byte aligned pieces
    return off;
  }
  size_t add_f(size_t n) {
    size_t off = f32.size();
    f32.resize(off + ((n + 31) / 32) * 32, 0.f);
    return off;
  }
};

// Hidden chunk c (c = 0..3) of a SwiGLU occupies rows [128c, 128c+64) = W1 rows [64c, 64c+64) and rows
// [128c+64, 128c+128) = W3 rows [64c, 64c+64): one N=128 MMA yields matching pre-activation columns. W1 and b1
// are stored halved (exact: a power of two), so the kernels get a / 2 for silu(a) = a/2 (1 + tanh(a/2)).
void pack_w13(uint16_t* dst, const float* w1, const float* w3, int din) {
  for (int c = 0; c < 4; ++c)
    for (int i = 0; i < 64; ++i)
      for (int k = 0; k < din; ++k) {
        dst[(size_t)(c * 128 + i) * din + k] = f32_to_bf16_bits(0.5f * bf16_round(w1[(size_t)(c * 64 + i) * din + k]));
        dst[(size_t)(c * 128 + 64 + i) * din + k] = f32_to_bf16_bits(w3[(size_t)(c * 64 + i) * din + k]);
      }
}
void pack_b13(float* dst, const float* b1, const float* b3) {
  for (int c = 0; c < 4; ++c)
    for (int i = 0; i < 64; ++i) {
      dst[c * 128 + i] = 0.5f * b1[c * 64 + i];
      dst[c * 128 + 64 + i] = b3[c * 64 + i];
    }
}

cvr_status free_workspace(cvr_handle* h) {
  for (auto& kv : h->graphs)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  h->graphs.clear();
  if (h->ws) cudaFree(h->ws);
  h->ws = nullptr;
  h->R_cap = h->B_cap = 0;
  return CVR_OK;
}

// merge counters of either attention kernel: one per (32-candidate tile, group), or one per (128-candidate
// tile, group, softmax warp)
size_t attn_count_bytes(int B_cap) {
  return std::max((size_t)(B_cap + 31) / 32 * kG, (size_t)(B_cap + 127) / 128 * kG * kAttnCounters) * 4;
}

// the per-block ready counters, one array: Token Mixer tiles per 128-row block, then attention groups per
// 32-candidate block
size_t ple_ready_words(int B_cap) { return (size_t)(B_cap + 127) / 128; }
size_t ready_bytes_of(int B_cap) { return (ple_ready_words(B_cap) + (size_t)(B_cap + 31) / 32) * 4; }

cvr_status ensure_workspace(cvr_handle* h, int R, int B) {
  if (R <= h->R_cap && B <= h->B_cap) return CVR_OK;
  free_workspace(h);
  const int R_cap = std::max(R, h->R_cap);
  const int B_cap = (int)(((int64_t)std::max(B, h->B_cap) + 127) / 128 * 128);
  int max_chunks = 0;
  for (int g = 0; g < kG; ++g) max_chunks = std::max(max_chunks, (h->L[g] + 511) / 512);  // column-sum blocks
  const int64_t seq_rows = (int64_t)R_cap * h->SL;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 1023) / 1024 * 1024;
    return o;
  };
  const int R_pad = (R_cap + 127) / 128 * 128;  // U is read by the tokeniser in 128-row tiles
  const size_t oU = take((size_t)R_pad * kUD * 2), oI = take((size_t)B_cap * kID * 2);
  const size_t oXs = take((size_t)seq_rows * kD * 2), oH = take((size_t)seq_rows * kD * 2);
  const size_t oCs = take((size_t)R_cap * kG * max_chunks * kD * 4), oXu = take((size_t)R_cap * kTokN * 4);
  const size_t oQb = take((size_t)h->n_layers * R_cap * kG * kD * 4);
  const size_t oZ = take((size_t)B_cap * kYD * 2), oY = take((size_t)B_cap * kYD * 2);
  const size_t oQ = take((size_t)B_cap * kG * kD * 2), oEx = take((size_t)B_cap * kPleN * 2);
  const size_t oG = take((size_t)B_cap * 8 * 4), oErr = take(1024), oCnt = take((size_t)R_cap * kG * 4);
  const size_t oReq = take((size_t)B_cap * 4);
  const size_t ready_bytes = ready_bytes_of(B_cap);  // Token Mixer tiles and attention groups written per block
  const size_t oRdy = take(ready_bytes);
  const size_t oR = take((size_t)2 * B_cap * kDE * 2);
  const size_t oXr = take((size_t)R_pad / 128 * (kTokN / 128) * 4);
  int splits = 1;
  for (int g = 0; g < kG; ++g) splits = std::max(splits, split_count(h->L[g]));
  // attention split state and merge counters, sized for either attention kernel: the register-tile one keeps
  // 20 floats per thread of 256 per 32-candidate tile, the tcgen05 one m[4], l[4], O[4][32] per row of a
  // 128-candidate tile and one counter per softmax warp
  const size_t st_bytes = std::max((size_t)(B_cap + 31) / 32 * kG * splits * 256 * 20 * 4,
                                   (size_t)(B_cap + 127) / 128 * kG * splits * 128 * kAttnStateFloats * 4);
  const size_t cnt_bytes = attn_count_bytes(B_cap);
  const size_t oAst = splits > 1 ? take(st_bytes) : 0;
  const size_t oAcnt = take(cnt_bytes);
  cudaError_t e = cudaMalloc(&h->ws, off);
  if (e != cudaSuccess) {
    h->ws = nullptr;
    cudaGetLastError();
    return fail(h, CVR_E_OOM, "workspace allocation failed: " + std::string(cudaGetErrorString(e)));
  }
  uint8_t* b = static_cast<uint8_t*>(h->ws);
  h->U = (bf16*)(b + oU);
  h->I = (bf16*)(b + oI);
  h->Xs = (bf16*)(b + oXs);
  h->H = (bf16*)(b + oH);
  h->colsum = (float*)(b + oCs);
  h->xu = (float*)(b + oXu);
  h->qb = (float*)(b + oQb);
  h->Z = (bf16*)(b + oZ);
  h->Y = (bf16*)(b + oY);
  h->Q = (bf16*)(b + oQ);
  h->Ex = (bf16*)(b + oEx);
  h->gates = (float*)(b + oG);
  h->err = (int*)(b + oErr);
  h->cs_count = (unsigned*)(b + oCnt);
  h->req_copy = (int32_t*)(b + oReq);
  h->ple_ready = (unsigned*)(b + oRdy);
  h->attn_ready = h->ple_ready + ple_ready_words(B_cap);
  h->Rt = (bf16*)(b + oR);
  h->xu_ready = (unsigned*)(b + oXr);
  h->attn_splits = splits;
  h->attn_state = splits > 1 ? (float*)(b + oAst) : nullptr;
  h->attn_count = (unsigned*)(b + oAcnt);
  e = cudaMemset(h->err, 0, 1024);  // the error word starts at zero; the host clears it after an error
  if (e == cudaSuccess) e = cudaMemset(h->cs_count, 0, (size_t)R_cap * kG * 4);  // reset by their last block
  if (e == cudaSuccess) e = cudaMemset(h->attn_count, 0, cnt_bytes);  // reset by the merging CTA or warp
  if (e == cudaSuccess) e = cudaMemset(h->ple_ready, 0, ready_bytes);  // (also cleared by every call's first kernel)
  if (e != cudaSuccess) {
    free_workspace(h);
    return fail(h, CVR_E_CUDA, "workspace initialisation failed");
  }
  h->R_cap = R_cap;
  h->B_cap = B_cap;
  h->max_chunks = max_chunks;
  bool ok = encode_2d(&h->tm_Xs, h->Xs, kD, (uint64_t)seq_rows, kD, 64, 128) &&
            encode_2d(&h->tm_I, h->I, kID, B_cap, kID, 64, 128) &&
            encode_2d(&h->tm_U, h->U, kUD, R_pad, kUD, 64, 128) &&
            encode_2d(&h->tm_U32, h->U, kUD, R_pad, kUD, 64, 32) &&
            encode_2d(&h->tm_x_Z, h->Z, kXD, B_cap, kYD, 64, 128) &&
            encode_2d(&h->tm_x_Y, h->Y, kXD, B_cap, kYD, 64, 128) &&
            encode_2d(&h->tm_full_Z, h->Z, kYD, B_cap, kYD, 64, 128) &&
            encode_2d(&h->tm_full_Y, h->Y, kYD, B_cap, kYD, 64, 128) &&
            encode_2d(&h->tm_Q, h->Q, kG * kD, B_cap, kG * kD, 64, 128) &&
            encode_2d(&h->tm_H, h->H, kD, (uint64_t)seq_rows, kD, 64, 64) &&
            encode_2d(&h->tm_R, h->Rt, kDE, (uint64_t)2 * B_cap, kDE, 64, 128) &&
            encode_2d(&h->tm_Ex, h->Ex, kPleN, B_cap, kPleN, 64, 128);
  if (!ok) {
    free_workspace(h);
    return fail(h, CVR_E_CUDA, "cuTensorMapEncodeTiled failed for a workspace tensor");
  }
  return CVR_OK;
}

constexpr int kMissCap = 1 << 20;  // rows a call can log for admission (more misses are served, not admitted)

int ilog2(int64_t v) {
  int k = 0;
  while ((int64_t(1) << k) < v) ++k;
  return k;
}

void free_cache(cvr_handle* h, int t) {
  for (void* p : {(void*)h->c_rows[t], (void*)h->c_tags[t], (void*)h->c_use[t], (void*)h->c_claim[t]})
    if (p) cudaFree(p);
  h->c_rows[t] = nullptr;
  h->c_tags[t] = nullptr;
  h->c_use[t] = nullptr;
  h->c_claim[t] = nullptr;
  h->c_slots[t] = 0;
}

void drop_graphs(cvr_handle* h) {
  for (auto& kv : h->graphs)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  h->graphs.clear();
}

FwdArgs make_args(cvr_handle* h, int R, int B, const int32_t* req_ids, const int64_t* bag_ids,
                  const int64_t* bag_offsets, const int64_t* seq_ids, float* out, float* dbg_pooled,
                  int64_t* dbg_rows) {
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.req_in = req_ids;
  a.req_ids = h->req_copy;
  a.req_copy = h->req_copy;
  a.bag_ids = bag_ids;
  a.bag_offsets = bag_offsets;
  a.seq_ids = seq_ids;
  a.out = out;
  a.dbg_pooled = dbg_pooled;
  a.dbg_rows = dbg_rows;
  for (int t = 0; t < kFu + kFi + 1; ++t) {
    a.tables[t] = h->tables[t];
    a.table_rows[t] = h->rows[t];
  }
  a.R = R;
  a.B = B;
  a.SL = h->SL;
  int64_t acc = 0;
  for (int g = 0; g < kG; ++g) {
    a.L[g] = h->L[g];
    a.goff[g] = acc;
    acc += (int64_t)R * h->L[g];
  }
  a.n_layers = h->n_layers;
  a.num_sms = h->num_sms;
  a.pdl = h->pdl ? 1 : 0;
  a.clamp = h->cfg.clamp;
  a.tau = h->cfg.tau;
  a.eps = h->cfg.rms_eps;
  a.U = h->U;
  a.I = h->I;
  a.Xs = h->Xs;
  a.H = h->H;
  a.colsum = h->colsum;
  a.cs_count = h->cs_count;
  for (int t = 0; t < kNTab; ++t) {
    if (!h->c_slots[t]) continue;
    a.cache_on = 1;
    a.cache_rows[t] = h->c_rows[t];
    a.cache_tags[t] = h->c_tags[t];
    a.cache_use[t] = h->c_use[t];
    a.cache_shift[t] = 64 - ilog2(h->c_slots[t]);
  }
  a.miss_list = h->miss_list;
  a.miss_cap = kMissCap;
  a.cache_ctl = h->cache_ctl;
  a.cache_stat = h->cache_stat;
  a.attn_state = h->attn_state;
  a.attn_count = h->attn_count;
  a.attn_splits = h->attn_splits;
  for (int g = 0; g < kG; ++g) a.g_order[g] = g;  // groups by padded length, longest first (stable)
  std::stable_sort(a.g_order, a.g_order + kG, [&](int x, int y) { return h->L[x] > h->L[y]; });
  a.max_chunks = h->max_chunks;
  a.xu = h->xu;
  a.xu_ready = h->xu_ready;
  a.qb = h->qb;
  a.Z = h->Z;
  a.Y = h->Y;
  a.Q = h->Q;
  a.Ex = h->Ex;
  a.gates = h->gates;
  a.ple_ready = h->ple_ready;
  // the register-tile attention counts its blocks for the Token Mixer (the tcgen05 one is waited for whole)
  a.attn_ready = h->attn_tc ? nullptr : h->attn_ready;
  a.Rt = h->Rt;
  a.err = h->err;
  a.err_host = h->err_host_dev;
  a.wblob = static_cast<const uint8_t*>(h->wblob);
  a.wblob_bytes = (int64_t)h->wblob_bytes;
  a.tokU = h->tokU;
  a.tok_b = h->tok_b;
  a.seq_b13 = h->seq_b13;
  a.seq_b2 = h->seq_b2;
  a.qm = h->qm;
  a.q_b = h->q_b;
  a.tm_b13 = h->tm_b13;
  a.tm_b2 = h->tm_b2;
  a.tm_gain = h->tm_gain;
  a.ple_b = h->ple_b;
  a.ple_s8 = h->ple_int8 ? h->ple_s8 : nullptr;
  a.keep_stages = h->keep_stages ? 1 : 0;
  a.head_b1 = h->head_b1;
  a.head_w2 = h->head_w2;
  a.head_b2 = h->head_b2;
  return a;
}

// Enqueues the whole forward pass on `s`. With `events`, records one after each kernel.
// Whether a call of R requests runs the tokeniser on the side stream, next to the sequence encoder: only when
// the encoder leaves at least half the SMs free, without per-kernel events and with the register-tile attention
// (which adds the first layer's mean-pooled query term the tokeniser then leaves out).
bool fork_tokenizer(const cvr_handle* h, int R, bool events) {
  int seq_tiles = 0;
  for (int g = 0; g < kG; ++g) seq_tiles += (int)(((int64_t)R * h->L[g] + 127) / 128);
  return !events && h->side && !h->attn_tc && std::min(seq_tiles, h->num_sms) <= h->num_sms / 2;
}

// CVR_STAGE_Q after such a call with one layer: the stored queries plus their mean-pooled term, rounded like
// the attention kernel rounds them
__global__ void q_with_mean_kernel(__nv_bfloat16* dst, const __nv_bfloat16* q, const float* qb, const int32_t* req,
                                   int64_t n, int R) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / (kG * kD);
    const int c = (int)(i - b * (kG * kD));
    const int r = min(max(req[b], 0), R - 1);
    dst[i] = __float2bfloat16_rn(__bfloat162float(q[i]) + qb[(int64_t)r * (kG * kD) + c]);
  }
}

cudaError_t enqueue_forward(cvr_handle* h, const FwdArgs& a, cudaStream_t s, bool events, bool external_events,
                            int* launches) {
  int n = 0, ev = 0;
  cudaError_t e = cudaSuccess;
  auto mark = [&](const char* name) {
    if (!events || e != cudaSuccess) return;
    if ((size_t)ev + 1 >= h->events.size()) return;
    h->event_names[ev] = name;
    e = external_events ? cudaEventRecordWithFlags(h->events[ev + 1], s, cudaEventRecordExternal)
                        : cudaEventRecord(h->events[ev + 1], s);
    ++ev;
  };
  auto run = [&](cudaError_t r, const char* name) {
    if (e != cudaSuccess) return;
    e = r;
    ++n;
    mark(name);
  };
  if (events)
    e = external_events ? cudaEventRecordWithFlags(h->events[0], s, cudaEventRecordExternal)
                        : cudaEventRecord(h->events[0], s);
  run(launch_sparse(a, s), kStageNames[0]);
  int seq_tiles = 0;
  for (int g = 0; g < kG; ++g) seq_tiles += (int)(((int64_t)a.R * a.L[g] + 127) / 128);
  const int seq_grid = std::min(seq_tiles, a.num_sms);
  // Two branches after the sparse kernel when the sequence encoder leaves at least half the SMs free. Side
  // stream: the tokeniser with its user row-tiles (it needs the pooled embeddings only), on the SMs the encoder
  // does not use. This stream: the sequence encoder and its column sums. The rest of the call then follows the
  // tokeniser on the side stream (the tokeniser ends last, so the attention launches on a programmatic edge from
  // it, with the column sums as a plain dependency) and joins this stream at the end. The first layer's queries
  // lack their mean-pooled sequence term, which the attention kernel adds (the tcgen05 attention reads Q by TMA
  // and keeps the one-stream order).
  const bool fork = fork_tokenizer(h, a.R, events);
  FwdArgs af = a;
  af.q_add = fork ? 1 : 0;
  cudaStream_t t = s;  // the stream of the attention and everything after it
  if (fork) {
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
    // (without a programmatic edge: its CTAs must not queue ahead of the encoder's for the SMs the gather frees)
    run(launch_tokenizer(af, h->tm_I, h->tm_tokI, h->tm_full_Z, h->tm_Q, h->tm_U, h->tm_U32, h->tm_tokU, a.num_sms - seq_grid,
                         false, h->side),
        kStageNames[3]);
    run(launch_seq_mlp(af, h->tm_Xs, h->tm_seqW13, h->tm_seqW2, seq_tiles, s), kStageNames[1]);
    // the column sums follow the encoder on a programmatic edge, which the encoder opens only as its last tiles
    // end: their CTAs wait for the SMs the encoder leaves, not on the SMs the tokeniser's CTAs need
    run(launch_seq_colsum(af, s), kStageNames[2]);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_join, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_join, 0);
    t = h->side;
  } else {
    run(launch_seq_mlp(a, h->tm_Xs, h->tm_seqW13, h->tm_seqW2, seq_tiles, s), kStageNames[1]);
    run(launch_seq_colsum(a, s), kStageNames[2]);
    run(launch_tokenizer(a, h->tm_I, h->tm_tokI, h->tm_full_Z, h->tm_Q, h->tm_U, h->tm_U32, h->tm_tokU, 0, true, s),
        kStageNames[3]);
  }
  bf16* zin = h->Z;
  bf16* zout = h->Y;
  for (int l = 0; l < a.n_layers; ++l) {
    if (l > 0) std::swap(zin, zout);  // layer l reads the previous output (its first 13 tokens) in place
    const bool in_is_Z = zin == h->Z;
    // the first layer's queries come out of the tokeniser
    if (l > 0) run(launch_query(a, l, in_is_Z ? h->tm_x_Z : h->tm_x_Y, h->tm_qW[l], h->tm_qWw[l], t), kStageNames[4]);
    FwdArgs al = a;  // the first layer's queries may still lack their mean-pooled term (stacked layers' have it)
    al.q_add = l == 0 ? af.q_add : 0;
    run(h->attn_tc ? launch_attention_tc(al, h->tm_Q, h->tm_H, zin, t) : launch_attention(al, zin, t), kStageNames[5]);
    run(launch_tm_mlp(a, l, zin, zout, h->tm_tmW13, h->tm_tmW2, t), kStageNames[6]);
  }
  run(launch_ple_heads(a, zout == h->Z ? h->tm_full_Z : h->tm_full_Y, h->ple_int8 ? h->tm_pleW8 : h->tm_pleW,
                       h->tm_R, h->tm_Ex, h->tm_headW1, h->B_cap, t),
      kStageNames[7]);
  if (a.cache_on) {
    run(launch_cache_admit(a, h->c_claim, t), kStageNames[8]);
    ++n;  // (two kernels)
  }
  if (fork) {  // the call ends on the handle's stream
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_tail, t);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_tail, 0);
  }
  h->last_zin = zin;
  h->last_zout = zout;
  if (launches) *launches = n;
  h->n_events_last = events ? ev : 0;
  return e;
}

cvr_status sync_status(cvr_handle* h);

cvr_status run_forward(cvr_handle* h, int32_t R, int32_t B, const int32_t* req_ids, const int64_t* bag_ids,
                       const int64_t* bag_offsets, const int64_t* seq_ids, float* out, float* dbg_pooled,
                       int64_t* dbg_rows, bool sync = true, const int32_t* seq_lens = nullptr) {
  if (!h) return CVR_E_ARG;
  if (!req_ids || !bag_ids || !bag_offsets || !seq_ids || !out) return fail(h, CVR_E_ARG, "null input or output pointer");
  if (R < 1 || B < 1 || R > 65535 || B > (1 << 20)) return fail(h, CVR_E_SHAPE, "need 1 <= n_req <= 65535, 1 <= n_cand <= 2^20");
  int cur = -1;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce == cudaSuccess && cur != h->device) ce = cudaSetDevice(h->device);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaSetDevice");
  cvr_status st = ensure_workspace(h, R, B);
  if (st != CVR_OK) return st;
  FwdArgs a = make_args(h, R, B, req_ids, bag_ids, bag_offsets, seq_ids, out, dbg_pooled, dbg_rows);
  a.seq_lens = seq_lens;
  cudaStream_t s = h->stream;
  if (h->use_graph) {
    std::vector<const void*> key = {req_ids, bag_ids, bag_offsets, seq_ids, seq_lens, out, dbg_pooled, dbg_rows,
                                    reinterpret_cast<const void*>((intptr_t)h->profile)};
    GraphEntry& ge = h->graphs[std::make_pair(R, B)];
    if (!ge.exec || ge.key != key) {
      cudaGraph_t graph = nullptr;
      ce = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
      if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaStreamBeginCapture");
      int launches = 0;
      cudaError_t le = enqueue_forward(h, a, h->cap_stream, h->profile, true, &launches);
      ce = cudaStreamEndCapture(h->cap_stream, &graph);
      if (le != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return cuda_fail(h, le, "kernel launch during capture");
      }
      if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaStreamEndCapture");
      bool updated = false;
      if (ge.exec) {
        cudaGraphExecUpdateResultInfo info;
        if (cudaGraphExecUpdate(ge.exec, graph, &info) == cudaSuccess) {
          updated = true;
        } else {
          cudaGetLastError();
          cudaGraphExecDestroy(ge.exec);
          ge.exec = nullptr;
        }
      }
      if (!updated) {
        ce = cudaGraphInstantiate(&ge.exec, graph, 0);
        if (ce != cudaSuccess) {
          cudaGraphDestroy(graph);
          ge.exec = nullptr;
          return cuda_fail(h, ce, "cudaGraphInstantiate");
        }
      }
      cudaGraphDestroy(graph);
      ge.key = key;
      ge.launches = launches;
    }
    ce = cudaGraphLaunch(ge.exec, s);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaGraphLaunch");
    h->last_launches = ge.launches;
    // the zin/zout bookkeeping of the captured sequence
    h->last_zin = (a.n_layers % 2 == 1) ? h->Z : h->Y;
    h->last_zout = (a.n_layers % 2 == 1) ? h->Y : h->Z;
  } else {
    int launches = 0;
    ce = enqueue_forward(h, a, s, h->profile, false, &launches);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "kernel launch");
    h->last_launches = launches;
  }
  h->last_R = R;
  h->last_kept = h->keep_stages;
  h->last_B = B;
  h->last_q_add = fork_tokenizer(h, R, h->profile) && h->n_layers == 1;
  if (!sync) return CVR_OK;
  return sync_status(h);
}

// Waits for the stream, then reads and clears the error bits every call since the last sync published.
cvr_status sync_status(cvr_handle* h) {
  cudaError_t ce = cudaStreamSynchronize(h->stream);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "forward pass");
  volatile int* hw = h->err_host;
  const int ew = *hw;
  *hw = 0;
  // the device word keeps its bits (every later call of the window reported them too): clear it for the next call
  if (ew && h->err) cudaMemset(h->err, 0, 4);
  if (ew & kErrTimeout) {
    // a CTA that gave up may have left a group or split counter part-way; the next call starts from zero
    if (h->cs_count) cudaMemset(h->cs_count, 0, (size_t)h->R_cap * kG * 4);
    if (h->attn_count) cudaMemset(h->attn_count, 0, attn_count_bytes(h->B_cap));
    if (h->ple_ready) cudaMemset(h->ple_ready, 0, ready_bytes_of(h->B_cap));
    return fail(h, CVR_E_TIMEOUT, "a bounded device-side wait gave up");
  }
  if (ew & kErrLayout) return fail(h, CVR_E_CUDA, "a kernel's shared-memory window was not 1024-byte aligned");
  if (ew & kErrSeqLens) return fail(h, CVR_E_INPUT, "a sequence length is outside [0, seq_len[g]]");
  if (ew & (kErrOffsets | kErrReqIds))
    return fail(h, CVR_E_INPUT, (ew & kErrOffsets) ? "bag offsets decrease" : "request ids out of range or decreasing");
  if (ew & kErrIdRange) return fail(h, CVR_E_ID_RANGE, "an id is outside its table (row 0 was read)");
  h->last_error.clear();
  return CVR_OK;
}

}  // namespace

// =============================================================================================
extern "C" {

const char* cvr_status_string(cvr_status s) {
  switch (s) {
    case CVR_OK: return "ok";
    case CVR_E_ARG: return "invalid argument";
    case CVR_E_SHAPE: return "size out of range";
    case CVR_E_ID_RANGE: return "id out of table range";
    case CVR_E_OOM: return "out of memory";
    case CVR_E_CUDA: return "CUDA error";
    case CVR_E_INPUT: return "invalid offsets or request ids";
    case CVR_E_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* cvr_last_error(const cvr_handle* h) { return h ? h->last_error.c_str() : "null handle"; }

int32_t cvr_last_launch_count(const cvr_handle* h) { return h ? h->last_launches : 0; }

cvr_status cvr_create(const cvr_weights* w, const cvr_config* cfg, void* cuda_stream, cvr_handle** out) {
  if (!out) return CVR_E_ARG;
  *out = nullptr;
  if (!w || !cfg) return CVR_E_ARG;
  std::string why;
  if (check_config(cfg, &why) != CVR_OK) {
    fprintf(stderr, "cvr_create: %s\n", why.c_str());
    return CVR_E_ARG;
  }
  const int NL = cfg->n_layers;
  // every pointer the configuration uses must be set
  bool ok = w->seq_table && w->tok_w && w->tok_b;
  for (int f = 0; f < 8; ++f) ok = ok && w->user_tables[f] && w->item_tables[f];
  for (int g = 0; g < 3; ++g)
    ok = ok && w->seq_w1[g] && w->seq_b1[g] && w->seq_w3[g] && w->seq_b3[g] && w->seq_w2[g] && w->seq_b2[g];
  for (int l = 0; l < NL; ++l) {
    for (int g = 0; g < 3; ++g) ok = ok && w->q_w[l][g] && w->q_b[l][g];
    ok = ok && w->tm_w1[l] && w->tm_b1[l] && w->tm_w3[l] && w->tm_b3[l] && w->tm_w2[l] && w->tm_b2[l] && w->tm_gain[l];
  }
  for (int k = 0; k < 3; ++k) ok = ok && w->ple_w[k] && w->ple_b[k];
  for (int t = 0; t < 2; ++t)
    ok = ok && w->gate_w[t] && w->gate_b[t] && w->head_w1[t] && w->head_b1[t] && w->head_w2[t] && w->head_b2[t];
  if (!ok) {
    fprintf(stderr, "cvr_create: a weight or table pointer is NULL\n");
    return CVR_E_ARG;
  }
  if (!get_encoder()) {
    fprintf(stderr, "cvr_create: cuTensorMapEncodeTiled is unavailable\n");
    return CVR_E_CUDA;
  }
  {
    cudaError_t pe = prepare_gemm_kernels();
    if (pe == cudaSuccess) pe = prepare_mlp_kernels();
    if (pe == cudaSuccess) pe = prepare_attention_kernel();
    if (pe == cudaSuccess) pe = prepare_attention_tc_kernel();
    if (pe == cudaSuccess) pe = prepare_ple_kernel();
    if (pe == cudaSuccess) pe = prepare_sparse_kernel();
    if (pe != cudaSuccess) {
      fprintf(stderr, "cvr_create: kernel attribute setup failed: %s\n", cudaGetErrorString(pe));
      cudaGetLastError();
      return CVR_E_CUDA;
    }
  }
  cvr_handle* h = new cvr_handle();
  h->cfg = *cfg;
  h->n_layers = NL;
  h->SL = 0;
  for (int g = 0; g < kG; ++g) {
    h->L[g] = cfg->seq_len[g];
    h->SL += cfg->seq_len[g];
  }
  cudaGetDevice(&h->device);
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (h->num_sms < 1) h->num_sms = 1;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  for (int f = 0; f < kFu; ++f) {
    h->tables[f] = w->user_tables[f];
    h->rows[f] = cfg->user_rows[f];
  }
  for (int f = 0; f < kFi; ++f) {
    h->tables[kFu + f] = w->item_tables[f];
    h->rows[kFu + f] = cfg->item_rows[f];
  }
  h->tables[kFu + kFi] = w->seq_table;
  h->rows[kFu + kFi] = cfg->seq_rows;

  // ---- pack dense weights ----
  Packer P;
  const size_t o_tokI = P.add_bf((size_t)kTokN * kID), o_tokU = P.add_bf((size_t)kTokN * kUD);
  const size_t o_seqW13 = P.add_bf((size_t)kG * 512 * kD), o_seqW2 = P.add_bf((size_t)kG * kD * kHid);
  const size_t o_qX = P.add_bf((size_t)NL * kG * kD * kXD), o_qm = P.add_bf((size_t)NL * kG * kD * kD);
  const size_t o_tmW13 = P.add_bf((size_t)NL * 512 * kD), o_tmW2 = P.add_bf((size_t)NL * kD * kHid);
  const size_t o_pleW = P.add_bf((size_t)kPleCols * kYD), o_headW1 = P.add_bf((size_t)kNT * kHH * kDE);
  const size_t f_tok_b = P.add_f(kTokN), f_seq_b13 = P.add_f(kG * 512), f_seq_b2 = P.add_f(kG * kD);
  const size_t f_q_b = P.add_f((size_t)NL * kG * kD), f_tm_b13 = P.add_f((size_t)NL * 512);
  const size_t f_tm_b2 = P.add_f((size_t)NL * kD), f_gain = P.add_f((size_t)NL * kD), f_ple_b = P.add_f(kPleCols + 32);
  const size_t f_hb1 = P.add_f(kNT * kHH), f_hw2 = P.add_f(kNT * kHH), f_hb2 = P.add_f(32);
  uint16_t* B = P.bf.data();
  float* F = P.f32.data();
  const int IN = kUD + kID;
  for (int n = 0; n < kXD; ++n)
    for (int k = 0; k < kUD; ++k) {
      B[o_tokU + (size_t)n * kUD + k] = f32_to_bf16_bits(w->tok_w[(size_t)n * IN + k]);
      B[o_tokI + (size_t)n * kID + k] = f32_to_bf16_bits(w->tok_w[(size_t)n * IN + kUD + k]);
    }
  std::memcpy(F + f_tok_b, w->tok_b, sizeof(float) * kXD);
  // The first layer's query FFN is linear in the tokens, so its token part folds into the tokeniser:
  // Wq_x (Wt_u u + Wt_i i + bt) = (Wq_x Wt_u) u + (Wq_x Wt_i) i + Wq_x bt. Rows 1664.. of the packed
  // tokeniser hold Wq_x Wt (from the bf16 weights, summed in double, rounded once to bf16) and Wq_x bt.
  {
    const int QIN0 = kXD + kD;
    std::vector<double> acc(IN);
    std::vector<float> wt_bf((size_t)kXD * IN);
    for (size_t i = 0; i < wt_bf.size(); ++i) wt_bf[i] = bf16_round(w->tok_w[i]);
    for (int g = 0; g < kG; ++g)
      for (int n = 0; n < kD; ++n) {
        const float* qrow = w->q_w[0][g] + (size_t)n * QIN0;
        std::fill(acc.begin(), acc.end(), 0.0);
        double bacc = 0.0;
        for (int c = 0; c < kXD; ++c) {
          const double qc = bf16_round(qrow[c]);
          if (qc == 0.0) continue;
          const float* wrow = wt_bf.data() + (size_t)c * IN;
          for (int k = 0; k < IN; ++k) acc[k] += qc * wrow[k];
          bacc += qc * w->tok_b[c];
        }
        const size_t row = (size_t)kXD + g * kD + n;
        for (int k = 0; k < kUD; ++k) B[o_tokU + row * kUD + k] = f32_to_bf16_bits((float)acc[k]);
        for (int k = 0; k < kID; ++k) B[o_tokI + row * kID + k] = f32_to_bf16_bits((float)acc[kUD + k]);
        F[f_tok_b + row] = (float)bacc;
      }
  }
  for (int g = 0; g < kG; ++g) {
    pack_w13(B + o_seqW13 + (size_t)g * 512 * kD, w->seq_w1[g], w->seq_w3[g], kD);
    for (size_t i = 0; i < (size_t)kD * kHid; ++i) B[o_seqW2 + (size_t)g * kD * kHid + i] = f32_to_bf16_bits(w->seq_w2[g][i]);
    pack_b13(F + f_seq_b13 + g * 512, w->seq_b1[g], w->seq_b3[g]);
    std::memcpy(F + f_seq_b2 + g * kD, w->seq_b2[g], sizeof(float) * kD);
  }
  const int QIN = kXD + kD;
  for (int l = 0; l < NL; ++l) {
    for (int g = 0; g < kG; ++g) {
      for (int n = 0; n < kD; ++n) {
        const float* row = w->q_w[l][g] + (size_t)n * QIN;
        for (int k = 0; k < kXD; ++k) B[o_qX + ((size_t)(l * kG + g) * kD + n) * kXD + k] = f32_to_bf16_bits(row[k]);
        for (int k = 0; k < kD; ++k) B[o_qm + ((size_t)(l * kG + g) * kD + n) * kD + k] = f32_to_bf16_bits(row[kXD + k]);
      }
      std::memcpy(F + f_q_b + (size_t)(l * kG + g) * kD, w->q_b[l][g], sizeof(float) * kD);
    }
    pack_w13(B + o_tmW13 + (size_t)l * 512 * kD, w->tm_w1[l], w->tm_w3[l], kD);
    for (size_t i = 0; i < (size_t)kD * kHid; ++i) B[o_tmW2 + (size_t)l * kD * kHid + i] = f32_to_bf16_bits(w->tm_w2[l][i]);
    pack_b13(F + f_tm_b13 + l * 512, w->tm_b1[l], w->tm_b3[l]);
    std::memcpy(F + f_tm_b2 + l * kD, w->tm_b2[l], sizeof(float) * kD);
    std::memcpy(F + f_gain + l * kD, w->tm_gain[l], sizeof(float) * kD);
  }
  std::vector<uint8_t> W8((size_t)kPleCols * kYD + (size_t)kPleCols * 4);
  // PLE rows in 4 slices of 208, one per CTA of a row block's cluster: slice n = units [64n, 64n + 64) of
  // experts 0, 1, 2, then the 6 gate rows (task-major), then 10 zero rows; biases in the same order
  for (int n = 0; n < 4; ++n) {
    for (int j = 0; j < 208; ++j) {
      const size_t row = (size_t)n * 208 + j;
      const float* src = nullptr;
      float bias = 0.f;
      if (j < kNE * 64) {
        const int k = j / 64, u = n * 64 + j % 64;
        src = w->ple_w[k] + (size_t)u * kYD;
        bias = w->ple_b[k][u];
      } else if (j < kNE * 64 + kNT * kNE) {
        const int t = (j - kNE * 64) / kNE, k = (j - kNE * 64) % kNE;
        src = w->gate_w[t] + (size_t)k * kYD;
        bias = w->gate_b[t][k];
      }
      for (int c = 0; c < kYD; ++c) B[o_pleW + row * kYD + c] = src ? f32_to_bf16_bits(src[c]) : 0;
      F[f_ple_b + row] = bias;
      // the same row in 8 bits: q = round-half-even(w / scale) with scale = max|w| / 127 (a zero row: q = 0, scale 0)
      double amax = 0.0;
      for (int c = 0; src && c < kYD; ++c) amax = std::max(amax, std::fabs((double)src[c]));
      const double sc = amax / 127.0;
      int8_t* q = reinterpret_cast<int8_t*>(W8.data()) + row * kYD;
      for (int c = 0; c < kYD; ++c) {
        const double v = sc > 0.0 ? std::nearbyint((double)src[c] / sc) : 0.0;
        q[c] = (int8_t)std::min(127.0, std::max(-127.0, v));
      }
      reinterpret_cast<float*>(W8.data() + (size_t)kPleCols * kYD)[row] = (float)sc;
    }
  }
  for (int t = 0; t < kNT; ++t) {
    for (size_t i = 0; i < (size_t)kHH * kDE; ++i) B[o_headW1 + (size_t)t * kHH * kDE + i] = f32_to_bf16_bits(w->head_w1[t][i]);
    std::memcpy(F + f_hb1 + t * kHH, w->head_b1[t], sizeof(float) * kHH);
    std::memcpy(F + f_hw2 + t * kHH, w->head_w2[t], sizeof(float) * kHH);
    F[f_hb2 + t] = w->head_b2[t][0];
  }
  const size_t bf_bytes = P.bf.size() * 2, f_bytes = P.f32.size() * 4;
  cudaError_t e = cudaMalloc(&h->wblob, bf_bytes + f_bytes);
  if (e != cudaSuccess) {
    delete h;
    cudaGetLastError();
    return CVR_E_OOM;
  }
  h->wblob_bytes = bf_bytes + f_bytes;
  uint8_t* wb = static_cast<uint8_t*>(h->wblob);
  e = cudaMemcpy(wb, P.bf.data(), bf_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(wb + bf_bytes, P.f32.data(), f_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&h->w8blob, W8.size());
  if (e == cudaSuccess) e = cudaMemcpy(h->w8blob, W8.data(), W8.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&h->err_host), 64, cudaHostAllocMapped);
  if (e == cudaSuccess) {
    *h->err_host = 0;
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->err_host_dev), h->err_host, 0);
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_tail, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cvr_destroy(h);
    cudaGetLastError();
    return CVR_E_CUDA;
  }
  bf16* wbf = reinterpret_cast<bf16*>(wb);
  float* wf = reinterpret_cast<float*>(wb + bf_bytes);
  h->tokI = wbf + o_tokI;
  h->tokU = wbf + o_tokU;
  h->seqW13 = wbf + o_seqW13;
  h->seqW2 = wbf + o_seqW2;
  h->qX = wbf + o_qX;
  h->qm = wbf + o_qm;
  h->tmW13 = wbf + o_tmW13;
  h->tmW2 = wbf + o_tmW2;
  h->pleW = wbf + o_pleW;
  h->headW1 = wbf + o_headW1;
  h->tok_b = wf + f_tok_b;
  h->seq_b13 = wf + f_seq_b13;
  h->seq_b2 = wf + f_seq_b2;
  h->q_b = wf + f_q_b;
  h->tm_b13 = wf + f_tm_b13;
  h->tm_b2 = wf + f_tm_b2;
  h->tm_gain = wf + f_gain;
  h->ple_b = wf + f_ple_b;
  h->ple_s8 = reinterpret_cast<float*>(static_cast<uint8_t*>(h->w8blob) + (size_t)kPleCols * kYD);
  h->head_b1 = wf + f_hb1;
  h->head_w2 = wf + f_hw2;
  h->head_b2 = wf + f_hb2;
  ok = encode_2d(&h->tm_seqW13, h->seqW13, kD, kG * 512, kD, 64, 256) &&
       encode_2d(&h->tm_seqW2, h->seqW2, kHid, kG * kD, kHid, 64, 128) &&
       encode_2d(&h->tm_tokI, h->tokI, kID, kTokN, kID, 64, 128) &&
       encode_2d(&h->tm_tokU, h->tokU, kUD, kTokN, kUD, 64, 128) &&
       encode_2d(&h->tm_tmW13, h->tmW13, kD, (uint64_t)NL * 512, kD, 64, 256) &&
       encode_2d(&h->tm_tmW2, h->tmW2, kHid, (uint64_t)NL * kD, kHid, 64, 128) &&
       encode_2d(&h->tm_pleW, h->pleW, kYD, kPleCols, kYD, 64, 208) &&
       encode_2d_u8(&h->tm_pleW8, h->w8blob, kYD, kPleCols, kYD, 64, 208) &&
       encode_2d(&h->tm_headW1, h->headW1, kDE, kNT * kHH, kDE, 64, 128);
  for (int l = 0; l < NL && ok; ++l)
    ok = encode_2d(&h->tm_qW[l], h->qX + (size_t)l * kG * kD * kXD, kXD, kG * kD, kXD, 64, kQryBNNarrow) &&
         encode_2d(&h->tm_qWw[l], h->qX + (size_t)l * kG * kD * kXD, kXD, kG * kD, kXD, 64, kQryBNWide);
  if (!ok) {
    cvr_destroy(h);
    return CVR_E_CUDA;
  }
  *out = h;
  return CVR_OK;
}

cvr_status cvr_score(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_ids,
                     const int64_t* bag_offsets, const int64_t* seq_ids, float* out) {
  return run_forward(h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, nullptr, nullptr);
}

cvr_status cvr_score_async(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_ids,
                           const int64_t* bag_offsets, const int64_t* seq_ids, float* out) {
  return run_forward(h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, nullptr, nullptr, false);
}
cvr_status cvr_score_varlen(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                            const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids,
                            const int32_t* seq_lens, float* out) {
  if (!seq_lens) return fail(h, CVR_E_ARG, "null seq_lens");
  return run_forward(h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, nullptr, nullptr, true, seq_lens);
}
cvr_status cvr_score_varlen_async(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                                  const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids,
                                  const int32_t* seq_lens, float* out) {
  if (!seq_lens) return fail(h, CVR_E_ARG, "null seq_lens");
  return run_forward(h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, nullptr, nullptr, false, seq_lens);
}

cvr_status cvr_sync(cvr_handle* h) {
  if (!h) return CVR_E_ARG;
  return sync_status(h);
}

cvr_status cvr_score_debug(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids,
                           const int64_t* bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids, float* out,
                           float* pooled_fp32, int64_t* rows) {
  return run_forward(h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, pooled_fp32, rows);
}

cvr_status cvr_score_host(cvr_handle* h, int32_t n_req, int32_t n_cand, const int32_t* req_ids, const int64_t* bag_ids,
                          int64_t n_bag_ids, const int64_t* bag_offsets, const int64_t* seq_ids, float* out) {
  if (!h) return CVR_E_ARG;
  if (!req_ids || !bag_ids || !bag_offsets || !seq_ids || !out) return fail(h, CVR_E_ARG, "null input or output pointer");
  if (n_req < 1 || n_cand < 1 || n_req > 65535 || n_cand > (1 << 20) || n_bag_ids < 0)
    return fail(h, CVR_E_SHAPE, "need 1 <= n_req <= 65535, 1 <= n_cand <= 2^20, n_bag_ids >= 0");
  cudaError_t ce = cudaSetDevice(h->device);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaSetDevice");
  const size_t b_req = (size_t)n_cand * 4, b_ids = (size_t)n_bag_ids * 8;
  const size_t b_off = ((size_t)n_req * kFu + (size_t)n_cand * kFi + 1) * 8;
  const size_t b_seq = (size_t)n_req * h->SL * kCols * 8, b_out = (size_t)n_cand * kNT * 4;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  // Arrays in pinned, device-mapped (or managed) host memory are read and written in place by the kernels
  // -- over NVLink-C2C on a Grace-Blackwell node this beats a staging copy; the others are staged.
  auto in_place = [](const void* ptr) -> void* {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (at.type == cudaMemoryTypeManaged) return const_cast<void*>(ptr);
    if (at.type == cudaMemoryTypeHost && at.devicePointer) return at.devicePointer;
    return nullptr;
  };
  const int32_t* z_req = (const int32_t*)in_place(req_ids);
  const int64_t* z_ids = b_ids ? (const int64_t*)in_place(bag_ids) : nullptr;
  const int64_t* z_off = (const int64_t*)in_place(bag_offsets);
  const int64_t* z_seq = (const int64_t*)in_place(seq_ids);
  float* z_out = (float*)in_place(out);
  const size_t need = al(b_req) + al(b_ids) + al(b_off) + al(b_seq) + al(b_out);
  if (need > h->stage_bytes) {
    // growing the staging area invalidates graphs that captured its addresses
    for (auto& kv : h->graphs)
      if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    h->graphs.clear();
    if (h->stage) cudaFree(h->stage);
    h->stage = nullptr;
    h->stage_bytes = 0;
    const size_t cap = need + need / 4;
    ce = cudaMalloc(&h->stage, cap);
    if (ce != cudaSuccess) {
      h->stage = nullptr;
      cudaGetLastError();
      return fail(h, CVR_E_OOM, "staging allocation failed");
    }
    h->stage_bytes = cap;
  }
  uint8_t* p = static_cast<uint8_t*>(h->stage);
  int32_t* d_req = (int32_t*)p;
  int64_t* d_ids = (int64_t*)(p + al(b_req));
  int64_t* d_off = (int64_t*)(p + al(b_req) + al(b_ids));
  int64_t* d_seq = (int64_t*)(p + al(b_req) + al(b_ids) + al(b_off));
  float* d_out = (float*)(p + al(b_req) + al(b_ids) + al(b_off) + al(b_seq));
  cudaStream_t s = h->stream;
  auto stage_in = [&](const void* src, void* dst, size_t bytes, const void* direct) -> const void* {
    if (direct) return direct;
    if (bytes && ce == cudaSuccess) ce = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s);
    return dst;
  };
  const int32_t* q_req = (const int32_t*)stage_in(req_ids, d_req, b_req, z_req);
  const int64_t* q_ids = (const int64_t*)stage_in(bag_ids, d_ids, b_ids, z_ids);
  const int64_t* q_off = (const int64_t*)stage_in(bag_offsets, d_off, b_off, z_off);
  const int64_t* q_seq = (const int64_t*)stage_in(seq_ids, d_seq, b_seq, z_seq);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "host-to-device input copy");
  cvr_status st = run_forward(h, n_req, n_cand, q_req, q_ids, q_off, q_seq, z_out ? z_out : d_out, nullptr, nullptr,
                              /*sync=*/false);
  if (!z_out) ce = cudaMemcpyAsync(out, d_out, b_out, cudaMemcpyDeviceToHost, s);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "device-to-host output copy");
  if (st != CVR_OK) {
    cudaStreamSynchronize(s);
    return st;
  }
  return sync_status(h);
}

cvr_status cvr_debug_stage(cvr_handle* h, int32_t stage, void* dst, int64_t bytes) {
  if (!h || !dst) return CVR_E_ARG;
  if (h->last_B == 0) return fail(h, CVR_E_ARG, "no call has run yet");
  const void* src = nullptr;
  int64_t need = 0;
  const int64_t B = h->last_B, R = h->last_R;
  switch (stage) {
    case CVR_STAGE_H: src = h->H; need = R * h->SL * kD * 2; break;
    case CVR_STAGE_Z: src = h->last_zin; need = B * kYD * 2; break;
    case CVR_STAGE_Q: src = h->Q; need = B * kG * kD * 2; break;
    case CVR_STAGE_Y: src = h->last_zout; need = B * kYD * 2; break;
    case CVR_STAGE_EXPERTS: src = h->Ex; need = B * kPleN * 2; break;
    case CVR_STAGE_GATES: src = h->gates; need = B * 8 * 4; break;
    default: return fail(h, CVR_E_ARG, "unknown stage");
  }
  if ((stage == CVR_STAGE_EXPERTS || stage == CVR_STAGE_GATES) && !h->last_kept)
    return fail(h, CVR_E_ARG, "the last call did not keep the expert outputs and gates (set CVR_OPT_KEEP_STAGES)");
  if (bytes != need) return fail(h, CVR_E_SHAPE, "stage size mismatch: expected " + std::to_string(need) + " bytes");
  cudaError_t ce = cudaSuccess;
  if (stage == CVR_STAGE_Q && h->last_q_add) {
    q_with_mean_kernel<<<h->num_sms * 4, 256, 0, h->stream>>>(static_cast<__nv_bfloat16*>(dst), h->Q, h->qb,
                                                               h->req_copy, B * kG * kD, (int)R);
    ce = cudaGetLastError();
  } else {
    ce = cudaMemcpyAsync(dst, src, (size_t)need, cudaMemcpyDeviceToDevice, h->stream);
  }
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(h->stream);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "stage copy");
  return CVR_OK;
}

cvr_status cvr_set_option(cvr_handle* h, int32_t option, int64_t value) {
  if (!h) return CVR_E_ARG;
  if (option == CVR_OPT_PROFILE) {
    const bool on = value != 0;
    if (on && h->events.empty()) {
      const int n = 2 + 5 + 3 * CVR_MAX_LAYERS + 2 + 4;
      h->events.resize(n);
      h->event_names.assign(n, nullptr);
      for (int i = 0; i < n; ++i) {
        cudaError_t e = cudaEventCreate(&h->events[i]);
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventCreate");
      }
    }
    h->profile = on;
    return CVR_OK;
  }
  if (option == CVR_OPT_CUDA_GRAPH) {
    h->use_graph = value != 0;
    return CVR_OK;
  }
  if (option == CVR_OPT_PDL || option == CVR_OPT_ATTENTION_TC || option == CVR_OPT_PLE_INT8 ||
      option == CVR_OPT_KEEP_STAGES) {
    if (option == CVR_OPT_PDL) h->pdl = value != 0;
    else if (option == CVR_OPT_ATTENTION_TC) h->attn_tc = value != 0;
    else if (option == CVR_OPT_PLE_INT8) h->ple_int8 = value != 0;
    else h->keep_stages = value != 0;
    drop_graphs(h);
    return CVR_OK;
  }
  return fail(h, CVR_E_ARG, "unknown option");
}

cvr_status cvr_stage_times(cvr_handle* h, float* ms, const char** names, int32_t cap, int32_t* n) {
  if (!h || !n) return CVR_E_ARG;
  *n = 0;
  if (!h->profile || h->n_events_last == 0) return fail(h, CVR_E_ARG, "profiling is off or no call was profiled");
  const int cnt = std::min<int>(cap, h->n_events_last);
  for (int i = 0; i < cnt; ++i) {
    float t = 0.f;
    cudaError_t e = cudaEventElapsedTime(&t, h->events[i], h->events[i + 1]);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventElapsedTime");
    if (ms) ms[i] = t;
    if (names) names[i] = h->event_names[i];
  }
  *n = cnt;
  return CVR_OK;
}

cvr_status cvr_cache_enable(cvr_handle* h, int32_t table, int64_t slots) {
  if (!h) return CVR_E_ARG;
  if (table < 0 || table >= kNTab) return fail(h, CVR_E_ARG, "table index outside [0, 17)");
  if (slots != 0 && (slots < 1024 || slots > (int64_t(1) << 28) || (slots & (slots - 1))))
    return fail(h, CVR_E_ARG, "cache slots must be 0 or a power of two in [1024, 2^28]");
  cudaError_t ce = cudaSetDevice(h->device);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(h->stream);  // no call in flight still reads the old cache
  if (ce == cudaSuccess && h->side) ce = cudaStreamSynchronize(h->side);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cache setup");
  free_cache(h, table);
  drop_graphs(h);  // captured calls hold the old cache's pointers
  if (slots == 0) return CVR_OK;
  if (!h->miss_list) {
    void* ctl = nullptr;
    ce = cudaMalloc(&h->miss_list, (size_t)kMissCap * 8);
    if (ce == cudaSuccess) ce = cudaMalloc(&ctl, 64);
    if (ce == cudaSuccess) ce = cudaMemset(ctl, 0, 64);
    const unsigned first_epoch = 1;  // slot epochs start at 0: no slot counts as read before its first hit
    if (ce == cudaSuccess) ce = cudaMemcpy((unsigned*)ctl + 1, &first_epoch, 4, cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) {
      if (h->miss_list) cudaFree(h->miss_list);
      if (ctl) cudaFree(ctl);
      h->miss_list = nullptr;
      cudaGetLastError();
      return fail(h, CVR_E_OOM, "cache miss log allocation failed");
    }
    h->cache_ctl = (unsigned*)ctl;
    h->cache_stat = (unsigned long long*)((uint8_t*)ctl + 16);
  }
  ce = cudaMalloc(&h->c_rows[table], (size_t)slots * kE * 4);
  if (ce == cudaSuccess) ce = cudaMalloc(&h->c_tags[table], (size_t)slots * 8);
  if (ce == cudaSuccess) ce = cudaMalloc(&h->c_use[table], (size_t)slots * 4);
  if (ce == cudaSuccess) ce = cudaMalloc(&h->c_claim[table], (size_t)slots * 4);
  if (ce == cudaSuccess) ce = cudaMemset(h->c_tags[table], 0xFF, (size_t)slots * 8);  // -1: empty
  if (ce == cudaSuccess) ce = cudaMemset(h->c_use[table], 0, (size_t)slots * 4);
  if (ce == cudaSuccess) ce = cudaMemset(h->c_claim[table], 0, (size_t)slots * 4);
  if (ce != cudaSuccess) {
    free_cache(h, table);
    cudaGetLastError();
    return fail(h, CVR_E_OOM, "cache allocation failed");
  }
  h->c_slots[table] = slots;
  return CVR_OK;
}

cvr_status cvr_cache_stats(cvr_handle* h, int64_t* hits, int64_t* misses) {
  if (!h || !hits || !misses) return CVR_E_ARG;
  *hits = *misses = 0;
  if (!h->cache_stat) return CVR_OK;
  unsigned long long v[2] = {0, 0};
  cudaError_t ce = cudaStreamSynchronize(h->stream);
  if (ce == cudaSuccess) ce = cudaMemcpy(v, h->cache_stat, 16, cudaMemcpyDeviceToHost);
  if (ce == cudaSuccess) ce = cudaMemset(h->cache_stat, 0, 16);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cache statistics");
  *hits = (int64_t)v[0];
  *misses = (int64_t)v[1];
  return CVR_OK;
}

void cvr_destroy(cvr_handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  if (h->stream) cudaStreamSynchronize(h->stream);
  if (h->side) cudaStreamSynchronize(h->side);  // (joins the handle's stream, unless a launch failed in between)
  free_workspace(h);
  for (int t = 0; t < kNTab; ++t) free_cache(h, t);
  if (h->miss_list) cudaFree(h->miss_list);
  if (h->cache_ctl) cudaFree(h->cache_ctl);
  if (h->stage) cudaFree(h->stage);
  if (h->wblob) cudaFree(h->wblob);
  if (h->w8blob) cudaFree(h->w8blob);
  if (h->err_host) cudaFreeHost(h->err_host);
  for (auto ev : h->events) cudaEventDestroy(ev);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->ev_tail) cudaEventDestroy(h->ev_tail);
  delete h;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Per-CTA timeline of the forward-pass kernels (a diagnostic of builds with -DCVR_TIMELINE).
#ifdef CVR_TIMELINE
namespace cvr {
__device__ unsigned long long g_timeline[kTlKernels * kTlCtas * 3];
}
#endif

extern "C" cvr_status cvr_timeline(cvr_handle* h, uint64_t* records, int64_t n_records, int32_t clear) {
  if (!h) return CVR_E_ARG;
#ifdef CVR_TIMELINE
  const int64_t total = (int64_t)kTlKernels * kTlCtas * 3;
  if (records && n_records != total)
    return fail(h, CVR_E_SHAPE, "cvr_timeline: records must hold " + std::to_string(total) + " values");
  cudaError_t ce = cudaStreamSynchronize(h->stream);
  if (ce == cudaSuccess && records) ce = cudaMemcpyFromSymbol(records, cvr::g_timeline, total * 8);
  if (ce == cudaSuccess && clear) {
    void* addr = nullptr;
    ce = cudaGetSymbolAddress(&addr, cvr::g_timeline);
    if (ce == cudaSuccess) ce = cudaMemset(addr, 0, total * 8);
    if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
  }
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cvr_timeline");
  return CVR_OK;
#else
  (void)records;
  (void)n_records;
  (void)clear;
  return fail(h, CVR_E_ARG, "cvr_timeline: this library was built without -DCVR_TIMELINE");
#endif
}

// ------------------------------------------------------------------------------------------
// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing arrives at, with the same wait
// the tensor-core kernels use; after its ~1 s limit the wait gives up, raises the timeout bit and the kernel
// publishes it like the last kernel of a call does. Nothing faults, traps or hangs.
namespace {
__global__ void selftest_wait_kernel(int* err, int* err_host) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  cta_sync();
  mbar_wait(&bar, 0, &abort_flag, err);
  cta_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    const int e = atomicExch(err, 0);
    volatile int* hw = err_host;
    *hw = *hw | e;
  }
}
}  // namespace

extern "C" cvr_status cvr_selftest_wait_timeout(cvr_handle* h) {
  if (!h) return CVR_E_ARG;
  int cur = -1;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce == cudaSuccess && cur != h->device) ce = cudaSetDevice(h->device);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaSetDevice");
  cvr_status st = ensure_workspace(h, 1, 1);  // the device error word
  if (st != CVR_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, h->stream>>>(h->err, h->err_host_dev);
  ce = cudaGetLastError();
  if (ce != cudaSuccess) return cuda_fail(h, ce, "self-test launch");
  return sync_status(h);
}

// ------------------------------------------------------------------------------------------
// Prediction step without allocation: the PLE and prediction-head kernel on a caller's Token Mixer
// output, its intermediate (the gate-weighted expert sums r_t) and the error word in one fixed file-scope
// device array instead of the handle's growable workspace.
namespace {

constexpr int kNoAllocMaxCand = CVR_NOALLOC_MAX_CAND;
constexpr size_t kNaROff = 0;                                                // r_t, bf16 [2][n][256]
constexpr size_t kNaErrOff = kNaROff + (size_t)2 * kNoAllocMaxCand * kDE * 2;
constexpr size_t kNaBytes = kNaErrOff + 512;                                 // error word (+0)
constexpr int kNaMaxDevices = 64;

std::mutex g_na_mu;
uint8_t* g_na_addr[kNaMaxDevices] = {};

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNaBytes];

namespace {

// Device address of the scratch array, looked up once per device.
cvr_status noalloc_scratch(cvr_handle* h, uint8_t** p) {
  std::lock_guard<std::mutex> lock(g_na_mu);
  if (h->device < 0 || h->device >= kNaMaxDevices) return fail(h, CVR_E_ARG, "device index out of range");
  if (!g_na_addr[h->device]) {
    void* addr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGetSymbolAddress of the prediction scratch");
    g_na_addr[h->device] = static_cast<uint8_t*>(addr);
  }
  *p = g_na_addr[h->device];
  return CVR_OK;
}

}  // namespace

extern "C" {

cvr_status cvr_predict_noalloc(cvr_handle* h, int32_t n_cand, const void* y, float* out) {
  if (!h) return CVR_E_ARG;
  if (!y || !out) return fail(h, CVR_E_ARG, "null Y or output pointer");
  if (n_cand < 0 || n_cand > kNoAllocMaxCand)
    return fail(h, CVR_E_SHAPE, "cvr_predict_noalloc takes 0 <= n_cand <= " + std::to_string(kNoAllocMaxCand) +
                                    " (its scratch is a fixed device array); got " + std::to_string(n_cand));
  if (reinterpret_cast<uintptr_t>(y) % 16 != 0) return fail(h, CVR_E_ARG, "Y must be 16-byte aligned");
  int cur = -1;
  cudaError_t ce = cudaGetDevice(&cur);
  if (ce == cudaSuccess && cur != h->device) ce = cudaSetDevice(h->device);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "cudaSetDevice");
  uint8_t* sc = nullptr;
  cvr_status st = noalloc_scratch(h, &sc);
  if (st != CVR_OK) return st;
  if (n_cand == 0) return CVR_OK;
  CUtensorMap tmY;
  if (!encode_2d(&tmY, y, kYD, (uint64_t)n_cand, kYD, 64, 128))
    return fail(h, CVR_E_CUDA, "cuTensorMapEncodeTiled failed for Y");
  FwdArgs a = make_args(h, 1, n_cand, nullptr, nullptr, nullptr, nullptr, out, nullptr, nullptr);
  // nothing but the prediction kernel's own buffers is reachable from these arguments
  a.U = a.I = a.Xs = a.H = a.Z = a.Y = a.Q = nullptr;
  a.colsum = a.xu = a.qb = nullptr;
  a.cs_count = nullptr;
  a.attn_state = nullptr;
  a.attn_count = nullptr;
  a.Ex = nullptr;  // the expert outputs and gates are not kept
  a.gates = nullptr;
  a.keep_stages = 0;
  a.Rt = reinterpret_cast<bf16*>(sc + kNaROff);
  a.ple_ready = nullptr;  // a caller's Y: the kernel waits for the preceding work in the stream instead
  a.attn_ready = nullptr;

  a.err = reinterpret_cast<int*>(sc + kNaErrOff);
  cudaStream_t s = h->stream;
  ce = cudaMemsetAsync(sc + kNaErrOff, 0, 512, s);  // the error word starts at zero
  CUtensorMap tmR;
  if (!encode_2d(&tmR, a.Rt, kDE, (uint64_t)2 * kNoAllocMaxCand, kDE, 64, 128))
    return fail(h, CVR_E_CUDA, "cuTensorMapEncodeTiled failed for the prediction scratch");
  // (the expert-output map is not used without keep_stages: r_t's map stands in for it)
  if (ce == cudaSuccess)
    ce = launch_ple_heads(a, tmY, h->ple_int8 ? h->tm_pleW8 : h->tm_pleW, tmR, tmR, h->tm_headW1, kNoAllocMaxCand, s);
  if (ce != cudaSuccess) return cuda_fail(h, ce, "prediction kernels");
  return sync_status(h);
}

}  // extern "C"
