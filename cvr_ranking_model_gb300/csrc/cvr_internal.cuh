// Internal definitions shared by the CVR scoring kernels: model constants, device error bits,
// the forward-pass argument block and thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor)
// and the 5th-generation tensor core (tcgen05 + TMEM) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cvr {

// ---- model dimensions (HyFormer-style CVR model of the iQIYI ad-CVR article, section 3.2) ----
constexpr int kFu = 8;            // user/context fields (one bag per request)
constexpr int kFi = 8;            // item fields (one bag per candidate)
constexpr int kE = 32;            // embedding width
constexpr int kNTab = 8 + 8 + 1;  // embedding tables: user fields, item fields, the shared sequence table
constexpr int kUD = kFu * kE;     // 256: user half of the non-sequence embedding
constexpr int kID = kFi * kE;     // 256: item half
constexpr int kN = 13;            // non-sequence tokens
constexpr int kD = 128;           // token_dim
constexpr int kG = 3;             // behaviour-sequence groups (= decoded tokens)
constexpr int kT = kN + kG;       // 16 tokens into the Token Mixer
constexpr int kXD = kN * kD;      // 1664
constexpr int kYD = kT * kD;      // 2048
constexpr int kTokN = kXD + kG * kD;  // 2048 tokeniser outputs: the 13 tokens + the first layer's 3 queries
constexpr int kCols = 4;          // id columns per sequence event
constexpr int kHid = 256;         // SwiGLU hidden width
constexpr int kHeads = 4;         // cross-attention heads
constexpr int kHD = kD / kHeads;  // 32
constexpr int kNE = 3;            // PLE experts
constexpr int kDE = 256;          // expert width
constexpr int kNT = 2;            // tasks
constexpr int kHH = 128;          // head hidden width
constexpr int kPleN = kNE * kDE;  // 768 expert columns
constexpr int kPleCols = 832;     // packed PLE rows: 4 slices of [3 x 64 expert units, 6 gate logits, 10 zero rows]
constexpr int kMaxLayers = 4;
// cross-attention over long sequences: a CTA takes at most kChunksPerSplit chunks of 64 positions; a
// group longer than that is split over up to kMaxSplits CTAs whose softmax states are merged
constexpr int kAttnChunk = 64, kChunksPerSplit = 8, kMaxSplits = 8;
constexpr int kAttnStateFloats = 2 * kHeads + kHeads * kHD;  // split state of one candidate row: m, l, O
constexpr int kAttnCounters = 8;  // merge counters per (128-candidate tile, group): one per softmax warp
__host__ __device__ constexpr int split_count(int L) {
  return L <= kAttnChunk * kChunksPerSplit ? 1
         : ((L + kAttnChunk * kChunksPerSplit - 1) / (kAttnChunk * kChunksPerSplit) < kMaxSplits
                ? (L + kAttnChunk * kChunksPerSplit - 1) / (kAttnChunk * kChunksPerSplit)
                : kMaxSplits);
}

// ---- device error word bits ----
constexpr int kErrIdRange = 1;      // a bag or sequence id outside its table
constexpr int kErrOffsets = 2;      // bag offsets not non-decreasing
constexpr int kErrReqIds = 4;       // request ids out of range or decreasing
constexpr int kErrTimeout = 8;      // a bounded wait in a tensor-core kernel gave up
constexpr int kErrDebugCap = 16;
constexpr int kErrLayout = 32;      // a kernel found its shared-memory window misaligned and did nothing
constexpr int kErrSeqLens = 64;     // a sequence length outside [0, L[g]]

// ---- arguments of the forward pass, one copy per call ----
struct FwdArgs {
  // caller inputs (device, or host memory the device reads in place)
  const int32_t* req_in;     // the caller's request ids, read once by the sparse kernel
  const int32_t* req_ids;    // their copy in the workspace, which every later kernel reads
  int32_t* req_copy;         // (the same copy, written by the sparse kernel)
  const int64_t* bag_ids;
  const int64_t* bag_offsets;
  const int64_t* seq_ids;
  float* out;
  // debug outputs (device, optional)
  float* dbg_pooled;
  int64_t* dbg_rows;
  // tables (device, borrowed)
  const float* tables[kFu + kFi + 1];
  int64_t table_rows[kFu + kFi + 1];
  // sizes
  int R, B, SL;
  int L[kG];
  int64_t goff[kG];   // first row of group g in the grouped sequence layout = R * (L0 + .. + L_{g-1})
  int n_layers;
  int num_sms;            // persistent-kernel grid size
  int pdl;                // launch with programmatic dependent launch
  float clamp, tau, eps;
  // workspace
  __nv_bfloat16* U;       // [R][256]
  __nv_bfloat16* I;       // [B][256]
  __nv_bfloat16* Xs;      // [sum_g R*L_g][128] sequence rows, group-major
  __nv_bfloat16* H;       // same layout: encoded sequence states
  float* colsum;          // [R][G][max_chunks][128] partial column sums of H (chunks of 512 positions)
  unsigned* cs_count;     // [R][G] blocks of the column-sum kernel done (zero between calls)
  const int32_t* seq_lens;  // [R][G] events each request really has per group, or null (all L[g])
  // partial softmax states of split sequences and the merge counters (zero between calls), laid out by the
  // attention kernel in use: register-tile kernel [B/32][G][splits][256 threads][20] and [B/32][G];
  // tcgen05 kernel [B/128][G][splits][128 rows][m 4, l 4, O 4x32] and [B/128][G][8 softmax warps]
  float* attn_state;
  unsigned* attn_count;
  int attn_splits;         // splits of the longest group (grid z of the attention kernel)
  int g_order[kG];         // attention grid row y runs group g_order[y]: longest sequences first, so that the
                           // CTAs that set the kernel's length are dispatched before the short ones
  int q_add;               // 1: Q holds the first layer's queries without their mean-pooled sequence term, which
                           // the attention kernel adds (the tokeniser ran before the sequence side finished)
  int max_chunks;
  float* xu;              // [R][2048] user half of the tokeniser and of the folded first-layer queries (no bias)
  unsigned* xu_ready;     // [R/128][16] user row-tiles of xu written by the tokeniser launch (zeroed every call)
  float* qb;              // [layers][R][384] per-request query term (+ bias)
  __nv_bfloat16* Z;       // [B][2048] interaction-layer buffers (ping-pong with Y)
  __nv_bfloat16* Y;       // [B][2048]
  __nv_bfloat16* Q;       // [B][384]
  __nv_bfloat16* Ex;      // [B][768] expert outputs (after ReLU)
  float* gates;           // [B][8] task gate probabilities (2 x 3, padded)
  int keep_stages;        // 1: the PLE also writes Ex and gates (read back by cvr_debug_stage); 0: skipped
  __nv_bfloat16* Rt;      // [2][rows][256] gate-weighted expert sums r_t (task-major), the heads' A operand
  unsigned* ple_ready;    // [B/128] per 128-row block: 8-candidate tiles the last Token Mixer has written, or null
                          // (zeroed by the first kernel of each call; null: wait for the previous grid instead)
  unsigned* attn_ready;   // [B/32] per 32-candidate block: groups whose decoded tokens the attention has written,
                          // summed over the layers (3 per layer), or null: the Token Mixer then waits for the whole
                          // attention grid (zeroed by the first kernel of each call)
  int* err;               // device error word (bits below), OR-ed by any kernel that finds an error; it keeps its
                          // bits until the host clears it after reporting them
  int* err_host;          // device view of a pinned host word: the last kernel's CTAs OR the error bits into it
  // hot-row cache in HBM in front of embedding tables (per table; null tags = no cache for that table)
  int cache_on;                      // any table has a cache
  const float* cache_rows[kNTab];      // [slots][32] fp32 copies of table rows
  const int64_t* cache_tags[kNTab];    // [slots] the id held by each slot, -1 = empty
  unsigned* cache_use[kNTab];          // [slots] epoch of the last call that read the slot
  int cache_shift[kNTab];              // slot = (id * golden) >> shift, slots = 2^(64 - shift)
  int64_t* miss_list;                // [miss_cap] (table << 48 | id) of rows that missed this call
  int miss_cap;
  unsigned* cache_ctl;               // [0] misses logged this call, [1] epoch of this call, [2] admit counter
  unsigned long long* cache_stat;    // [0] hits, [1] misses, accumulated until read
  // packed weights (device): one allocation, which the first kernel of a call prefetches into L2
  const uint8_t* wblob;
  int64_t wblob_bytes;
  const __nv_bfloat16* tokU;   // [1664][256]
  const float* tok_b;          // [1664]
  const float* seq_b13;        // [3][512] (interleaved like the weights)
  const float* seq_b2;         // [3][128]
  const __nv_bfloat16* qm;     // [layers][3][128][128]: query weights applied to the mean-pooled sequence
  const float* q_b;            // [layers][384]
  const float* tm_b13;         // [layers][512]
  const float* tm_b2;          // [layers][128]
  const float* tm_gain;        // [layers][128]
  const float* ple_b;          // [4][208]: biases of the PLE slices (3 x 64 expert units, 6 gates, zeros)
  const float* ple_s8;         // [4][208]: row scales of the 8-bit PLE weights, or null (bf16 weights)
  const float* head_b1;        // [2][128]
  const float* head_w2;        // [2][128]
  const float* head_b2;        // [2]
};

// ------------------------------------------------------------------------------------------
// Per-CTA timeline (builds with -DCVR_TIMELINE only; a diagnostic, off in the normal build): the first thread of every
// CTA of the forward-pass kernels records %globaltimer at entry, when its dependency wait returned and at exit, in
// g_timeline[kernel id][CTA][3]; cvr_timeline copies the last call's records out.
constexpr int kTlKernels = 10, kTlCtas = 8192;
enum { TL_SPARSE = 0, TL_SEQ_MLP = 1, TL_COLSUM = 2, TL_TOKENIZER = 3, TL_QUERY = 4, TL_ATTENTION = 5,
       TL_TOKEN_MIXER = 6, TL_PLE_HEADS = 7, TL_ATTENTION_TC = 8 };
#ifdef CVR_TIMELINE
extern __device__ unsigned long long g_timeline[kTlKernels * kTlCtas * 3];
struct TimelineCta {
  unsigned slot;
  __device__ explicit TimelineCta(int kernel) {
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    slot = cta < (unsigned)kTlCtas ? ((unsigned)kernel * kTlCtas + cta) * 3 : 0xffffffffu;
    if (threadIdx.x == 0 && slot != 0xffffffffu) g_timeline[slot] = stamp();
  }
  __device__ void waited() const {
    if (slot != 0xffffffffu) g_timeline[slot + 1] = stamp();
  }
  __device__ ~TimelineCta() {
    if (threadIdx.x == 0 && slot != 0xffffffffu) g_timeline[slot + 2] = stamp();
  }
  __device__ static unsigned long long stamp() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
  }
};
#define CVR_TL_BEGIN(kernel) const TimelineCta cvr_tl_(kernel)
#define CVR_TL_WAITED() cvr_tl_.waited()
#else
#define CVR_TL_BEGIN(kernel) ((void)0)
#define CVR_TL_WAITED() ((void)0)
#endif

// ------------------------------------------------------------------------------------------
// inline PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after ~1 s, raises the CTA's abort flag and the device error word.
// Every wait of a CTA checks the abort flag first, so one timeout ends the whole CTA quickly.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > 1000000000ull) {
      *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
// The same wait taken by a whole warp, with one answer for all of its lanes: code that follows it with
// warp-collective instructions (tcgen05.ld/st) never runs with part of the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}
// After an abort: wait (bounded, ignoring the abort flag) for copies or MMAs this CTA itself issued, so that
// none lands in shared memory or TMEM after they are released.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 1000000000ull) return false;
  return true;
}
// Events that request r really has in group g (variable-length sequences); kept in [0, L[g]] so that no
// access ever leaves the padded layout (the sparse kernel reports a value outside that range).
__device__ __forceinline__ int seq_len_of(const FwdArgs& a, int64_t r, int g) {
  if (!a.seq_lens) return a.L[g];
  const int v = a.seq_lens[r * kG + g];
  return v < 0 ? 0 : (v > a.L[g] ? a.L[g] : v);
}
// Programmatic dependent launch: let the next kernel in the stream launch (its prologue overlaps this
// kernel), and wait until the previous kernel has completed and its writes are visible. Every kernel of
// the forward pass waits before touching data an earlier kernel wrote, which keeps the ordering transitive.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tiled loads into shared memory, completing on an mbarrier (transaction bytes)
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// TMA tiled store shared -> global (bulk-group completion): the box at (x, y) of `map` from `src`
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed store groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until every committed store group has completed (written to global memory)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int x0, int x1, int x2,
                                            int x3, int x4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, "
      "%7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(x4)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 / TMEM ----
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Shared-memory matrix descriptors (tcgen05 format, version 1).
// K-major, 128-byte swizzle: rows of 128 B, 8-row atoms 1024 B apart (tile base 1024-B aligned).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// K-major, no swizzle: 8x16-byte core matrices; lbo = byte step between core matrices along K,
// sbo = byte step between 8-row groups along M/N.
__device__ __forceinline__ uint64_t sdesc_noswz(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46);
}
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M=128 rows = lanes, 16-bit elements packed two per column) read
// from tensor memory, issued by one thread
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// mbarrier arrives once every previously issued tcgen05.mma of this thread has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base lane + i). The _nowait form
// leaves the registers pending until tmem_ld_wait(), so several loads can be in flight at once.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive fp32 columns (see tmem_ld32_nowait)
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns from registers (thread i -> lane base + i)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns from registers
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  tmem_ld32_nowait(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// silu(x) = x * sigmoid(x) = x * (0.5 + 0.5 tanh(x / 2)): one MUFU op (tanh.approx) per value
__device__ __forceinline__ float silu_tanh(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return x * fmaf(0.5f, t, 0.5f);
}

// 32 consecutive fp32 values (16-byte aligned, read-only for the kernel) into registers, issued together
__device__ __forceinline__ void ldg32(const float* p, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = __ldg(q + i);
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
}

// 32 consecutive fp32 values through L2 (data written earlier in the same launch by another CTA)
__device__ __forceinline__ void ldcg32(const float* p, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = __ldcg(q + i);
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
}
// CTA barrier taken by converged warps: bar.sync expects every lane of a warp to arrive together, and single
// lanes of a warp (a producer or MMA-issuing thread, a thread that publishes a counter) often arrive after a
// branch of their own
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}
// counter publication: a release at GPU scope (orders this thread's earlier writes, and by cumulativity those of
// threads it synchronised with through a CTA barrier, before the increment)
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits (at most ~1 s) until *cnt >= need; a wait that gives up is reported and the caller goes on (every access
// stays in bounds whatever the data), so nothing can hang on a producer that never finishes.
__device__ __forceinline__ void wait_count(const unsigned* cnt, unsigned need, int* err) {
  if (ld_acquire_u32(cnt) >= need) return;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u32(cnt) < need) {
    if (global_timer_ns() - t0 > 1000000000ull) {
      atomicOr(err, kErrTimeout);
      return;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// Packed fp32 pairs (Blackwell f32x2 ALU ops): two values per instruction.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// silu(a) * g for two pairs at once, given h = a / 2 (the first SwiGLU weights and bias are stored halved):
// silu(a) g = a sigmoid(a) g = h g (1 + tanh(h)). Both tanh values come from one tanh.approx.f16x2 (the multi-
// function unit, the epilogues' narrowest pipe, then does one op per pair); its half-precision error is below the
// bf16 rounding of the result. Returns bf16x2 (round to nearest even).
__device__ __forceinline__ uint32_t silu_half_mul_bf16x2(uint64_t h, uint64_t g) {
  uint32_t hh, th;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hh) : "f"(__uint_as_float((uint32_t)(h >> 32))), "f"(__uint_as_float((uint32_t)h)));
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(th) : "r"(hh));
  float t0, t1;
  asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.f32.f16 %0, lo;\n cvt.f32.f16 %1, hi;\n}" : "=f"(t0), "=f"(t1) : "r"(th));
  const uint64_t hg = mul_f32x2(h, g);
  const uint64_t r = fma_f32x2(hg, f2pack(t0, t1), hg);
  return pack_bf16(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
// byte offset of 16-byte chunk `c` of row `r` inside a 128B-swizzled K-major tile (rows of 128 B)
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------------------------------
// Launch with the programmatic-stream-serialization attribute when `pdl` (the first kernel of a sequence
// is launched without it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// kernel launchers (each returns the launch's error code)
cudaError_t prepare_gemm_kernels();  // shared-memory attributes; once per device before any launch
cudaError_t prepare_mlp_kernels();
cudaError_t prepare_attention_kernel();
cudaError_t prepare_attention_tc_kernel();
cudaError_t launch_sparse(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_seq_colsum(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_seq_mlp(const FwdArgs& a, const CUtensorMap& tmXs, const CUtensorMap& tmW13,
                           const CUtensorMap& tmW2, int n_tiles, cudaStream_t s);
// the Token Mixer of layer `layer`: zin [B][16][128] -> yout
cudaError_t launch_tm_mlp(const FwdArgs& a, int layer, const __nv_bfloat16* zin, __nv_bfloat16* yout,
                          const CUtensorMap& tmW13, const CUtensorMap& tmW2, cudaStream_t s);
// the tokeniser GEMM (13 tokens + the first layer's queries, 2048 packed columns) on at most max_grid CTAs (0: one
// per SM). The user half xu comes from U with the user weights tmWu: with at most 32 requests every CTA computes
// its own column tile's slice (tmU32: U in boxes of 32 rows, tmWu as the A operand); else the launch's first
// M-tiles compute it (tmU: boxes of 128 rows). pdl = false launches it after the previous work in the stream has
// completed (the first kernel of the side stream).
cudaError_t launch_tokenizer(const FwdArgs& a, const CUtensorMap& tmI, const CUtensorMap& tmW, const CUtensorMap& tmZo,
                             const CUtensorMap& tmQo, const CUtensorMap& tmU, const CUtensorMap& tmU32,
                             const CUtensorMap& tmWu, int max_grid, bool pdl, cudaStream_t s);
// Requests up to which each tokeniser CTA computes its own column tile's user half.
constexpr int kTokOwnXuMaxR = 32;
// Columns of Q per tile of the stacked layers' query GEMM, narrow or wide (launch_query picks one per batch); also
// the row counts of the boxes of its two weight tensor maps.
constexpr int kQryBNNarrow = 96, kQryBNWide = 128;
// tmW: the layer's weights with boxes of kQryBNNarrow rows, tmWw with boxes of kQryBNWide rows
cudaError_t launch_query(const FwdArgs& a, int layer, const CUtensorMap& tmX, const CUtensorMap& tmW,
                         const CUtensorMap& tmWw, cudaStream_t s);
cudaError_t launch_attention(const FwdArgs& a, __nv_bfloat16* zin, cudaStream_t s);
cudaError_t launch_attention_tc(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmH, __nv_bfloat16* zin,
                                cudaStream_t s);
cudaError_t prepare_ple_kernel();
cudaError_t prepare_sparse_kernel();
// PLE experts, gates and r_t (four CTAs per 128-row block), then the heads of each block in its last CTA;
// tmW = packed PLE slices [832][2048], tmR = R viewed as [2 * r_rows][256], tmEx = expert outputs [rows][768],
// tmW1 = head first layers [2 * 128][256] (boxes of 64 x 128 like the others; all 128-byte swizzle); launched as
// clusters of four CTAs
cudaError_t launch_ple_heads(const FwdArgs& a, const CUtensorMap& tmY, const CUtensorMap& tmW, const CUtensorMap& tmR,
                             const CUtensorMap& tmEx, const CUtensorMap& tmW1, int r_rows, cudaStream_t s);
// hot-row cache admission after a call: rows that missed replace their slot's row unless that row was read
// in the same call; claims [kNTab] are the per-table election arrays (zero between calls)
cudaError_t launch_cache_admit(const FwdArgs& a, unsigned* const* claims, cudaStream_t s);

}  // namespace cvr
