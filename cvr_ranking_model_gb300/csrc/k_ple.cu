// PLE experts, task gates and prediction heads of the CVR forward pass (iQIYI ad-CVR article, section 3.2.4:
// three single-layer experts over the flattened tokens, a softmax gate per task, and per task a two-layer head
// ending in a sigmoid pCVR).
//
//  ple_kernel    four CTAs per 128-row block. CTA n computes, for the block's rows, the 208 columns
//                  [e_0 units 64n..64n+63 | e_1 units .. | e_2 units .. | the 6 gate logits | 10 zero columns]
//                of Y . W^T (Y [rows][2048] bf16, K = 2048) on tcgen05 with the accumulator in TMEM, A and B
//                streamed by TMA through a 5-stage mbarrier ring. Every CTA has all gate logits, so each forms
//                its 64-unit slice of r_t = sum_k g_t[k] ReLU(e_k + b_k) for both tasks (fp32, then bf16) and
//                writes it with TMA stores into R [task][row][256] (and, when the call keeps them, the expert
//                outputs and the gates).
//  heads         the four CTAs of a row block form a cluster. Once all four slices of R are written (one cluster
//                barrier), CTAs 2t and 2t + 1 both compute task t's hidden layer ReLU(W1_t r_t + b1) on tcgen05
//                (M=128, N=128, K=256) with r_t read back through L2 and W1_t loaded into the ring, apply the
//                128 -> 1 layer in two halves of 64 units added in shared memory, and finish (bias, sigmoid) rows
//                [0, 64) and [64, 128) of the block respectively: no partial sum crosses CTAs.
//
// The kernel starts per row block instead of waiting for the whole Token Mixer grid: a CTA waits (bounded)
// until the Token Mixer has counted every tile of its row block as written, so the first blocks run on the SMs
// the Token Mixer's last round leaves free. The counters are cleared by the first kernel of every call.
// INT8 weights (ple_kernel<true>): the expert and gate rows are held as signed 8-bit integers q with one fp32
// scale per row (W ~ scale . q, scale = max|W_row| / 127). The scale is constant along K, so it comes out of the
// dot product: the ring brings in q, the epilogue warps turn each stage into exact bf16 integers in the
// B operand's swizzled layout while the MMAs of earlier stages run, and the epilogue multiplies the fp32 sums by
// the row scales before the bias. The ring has 4 stages in this mode (the 8-bit staging takes the fifth's room).
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kSlice = 64;                  // units of each expert per CTA
constexpr int kSlices = kDE / kSlice;       // 4 CTAs per 128-row block
constexpr int kBN = kNE * kSlice + 16;      // 208 columns per CTA: 3 x 64 expert units + 16 gate columns
constexpr int kGateCol = kNE * kSlice;      // 192: the 6 gate logits (task-major), then zero columns
constexpr int kBM = 128, kBK = 64;
constexpr int kATile = kBM * kBK * 2;       // 16 KB
constexpr int kBTile = kBN * kBK * 2;       // 26 KB
constexpr int kW8Tile = kBN * kBK;          // 13 KB: one stage of 8-bit weights (rows of 64 bytes, unswizzled)
constexpr int kNK = kYD / kBK;              // 32 k-blocks
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..9 epilogue
constexpr int kTmemCols = 256;
constexpr int kHN = kHH;                    // hidden units per CTA: all of its task's (the CTA pair of a task
                                            // computes them twice and finishes half the rows each)
constexpr int kHOffW = 4 * kATile;
constexpr int kHBytes = 4 * kATile + 4 * kHN * kBK * 2;  // 128 KB
static_assert(kPleCols == kSlices * kBN, "four 208-column slices");

// shared memory (offsets from a 1024-byte aligned base)
template <bool I8>
struct Smem {
  static constexpr int kStages = I8 ? 4 : 5;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kStages * kATile;
  static constexpr int kOffW8 = kOffB + kStages * kBTile;  // (8-bit weights only)
  static constexpr int kRingBytes = kStages * (kATile + kBTile + (I8 ? kW8Tile : 0));
  // output staging, in the ring once the main loop is done: r_t slices [task] then expert slices [k], each
  // [128 rows][64 units] bf16 with the 128-byte swizzle (the layout of a TMA box of 64 x 128); the heads' operands
  // (r_t as 4 K-blocks of [128][64], then this CTA's W1 rows as 4 K-blocks of [64][64]) go there as well
  static constexpr int kOffStage = 0;
  static constexpr int kOffBias = kRingBytes;                   // fp32 slice bias [208], head b1 / w2 of this half [64] each
  static constexpr int kOffScale = kOffBias + (kBN + 2 * kHN) * 4;  // fp32 row scales of the slice [208] (8-bit weights)
  static constexpr int kOffPlog = kOffScale + (I8 ? kBN * 4 : 0);   // fp32 [2 halves][128 rows]: partial logits
  static constexpr int kOffBar = kOffPlog + 2 * kBM * 4;
  // per stage: full, empty (and for 8-bit weights: converted, weights landed); then acc_full, h_full, head_full,
  // w1_full
  static constexpr int kNBar = 4 * kStages + 4;
  static constexpr int kBytes = kOffBar + kNBar * 8 + 16 + 1024;  // + alignment slack
  static_assert((kNT + kNE) * kATile <= kRingBytes, "output staging fits the ring");
  static_assert(kHBytes <= kRingBytes, "head operands fit the ring");
  static_assert(kOffB % 1024 == 0 && kBTile % 1024 == 0 && kOffW8 % 1024 == 0, "stage alignment");
  static_assert(kBytes <= 232448, "shared memory budget of one CTA");
};

// 16 signed bytes (K order) -> 16 bf16 holding the same integers (exact: |q| <= 128 needs 8 significant bits).
// Each byte, biased to unsigned, becomes the low mantissa byte of the fp32 2^23 + u; subtracting 2^23 + 128 gives q.
__device__ __forceinline__ void s8x16_to_bf16(const uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float f0 = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7440u + 2 * h)) - 8388736.f;
      const float f1 = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7441u + 2 * h)) - 8388736.f;
      o[2 * i + h] = pack_bf16(f0, f1);
    }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// every thread of every CTA of the cluster arrives; memory before it (shared and global) is visible after it
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}

template <bool I8>
__global__ void __launch_bounds__(kThreads, 1)
    ple_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmY,
               const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmR,
               const __grid_constant__ CUtensorMap tmEx, const __grid_constant__ CUtensorMap tmW1, int r_rows) {
  using S = Smem<I8>;
  constexpr int kStages = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  CVR_TL_BEGIN(TL_PLE_HEADS);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sbias = reinterpret_cast<float*>(smem + S::kOffBias);  // [208]
  float* sb1 = sbias + kBN;                                  // [128]
  float* sw2 = sb1 + kHN;                                    // [128]
  float* sscale = reinterpret_cast<float*>(smem + S::kOffScale);  // [208] (8-bit weights)
  float* plog = reinterpret_cast<float*>(smem + S::kOffPlog);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* full = bar;
  uint64_t* empty = bar + kStages;
  uint64_t* acc_full = bar + 2 * kStages;  // the main loop's accumulator is complete
  uint64_t* h_full = acc_full + 1;         // heads: r_t (and the W1 rows when they come late) landed
  uint64_t* head_full = acc_full + 2;      // heads: hidden pre-activations complete
  uint64_t* w1_full = acc_full + 3;        // heads: the W1 rows landed (loaded right after the main loop)
  uint64_t* conv = acc_full + 4;           // 8-bit weights: stage s turned into bf16 by the epilogue warps
  uint64_t* wfull = conv + kStages;        // 8-bit weights: stage s's bytes landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + S::kNBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = (int)blockIdx.x % kSlices;            // slice of this CTA (= its rank in the cluster)
  const int rb = (int)blockIdx.x / kSlices;           // row block
  const int m0 = rb * kBM;
  const int ht = n >> 1, hh = n & 1;                  // head task of this CTA and the half of the rows it finishes
  const bool w1_early = !a.keep_stages;
  static_assert(kNT * kATile <= kHOffW, "the staged r_t slices end before the W1 rows");
  bool w1_issued = false;  // (warp 0, lane 0)
  int err_seen = 0;        // (thread 0) the error word after every earlier kernel has completed
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if constexpr (I8) {
        mbar_init(&conv[s], kEpiWarps);
        mbar_init(&wfull[s], 1);
      }
    }
    mbar_init(acc_full, 1);
    mbar_init(h_full, 1);
    mbar_init(head_full, 1);
    mbar_init(w1_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmY);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmR);
    tma_prefetch_desc(&tmEx);
    tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // weights first: they do not depend on the Token Mixer. 8-bit weights land in the staging area on their own
      // barrier, so that the epilogue warps convert the first stages while the activations are awaited.
      constexpr int kWBytes = I8 ? kW8Tile : kBTile;
      uint8_t* wdst = smem + (I8 ? S::kOffW8 : S::kOffB);
      uint64_t* wbar = I8 ? wfull : full;
      const int pre = kStages < kNK ? kStages : kNK;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_expect_tx(&full[kb], I8 ? kATile : kATile + kBTile);
        if constexpr (I8) mbar_expect_tx(&wfull[kb], kW8Tile);
        tma_load_2d(wdst + kb * kWBytes, &tmW, &wbar[kb], kb * kBK, n * kBN);
      }
      // then this row block's activations, once the Token Mixer has written every one of its 8-candidate tiles;
      // without the counters (a caller's Y) the previous work in the stream is waited for
      if (a.ple_ready) {
        wait_count(a.ple_ready + rb, (unsigned)((min(kBM, a.B - m0) + 7) / 8), a.err);
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the rows are read by TMA (async proxy)
        CVR_TL_WAITED();
      } else {
        pdl_wait();
      }
      for (int kb = 0; kb < kNK; ++kb) {
        const int s = kb % kStages;
        if (kb >= kStages) {
          if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag, a.err)) break;
          mbar_expect_tx(&full[s], I8 ? kATile : kATile + kBTile);
          if constexpr (I8) mbar_expect_tx(&wfull[s], kW8Tile);
          tma_load_2d(wdst + s * kWBytes, &tmW, &wbar[s], kb * kBK, n * kBN);
        }
        tma_load_2d(smem + S::kOffA + s * kATile, &tmY, &full[s], kb * kBK, m0);
      }
      // the heads' W1 rows: into the ring as soon as the main loop's MMAs have read it, so that they land during
      // the epilogue and the r_t exchange (the staged r_t slices use the ring's first 32 KB only; staged expert
      // outputs would reach the W1 area, so with those the rows come after the cluster barrier)
      if (w1_early && mbar_wait(acc_full, 0, abort_flag, a.err)) {
        mbar_expect_tx(w1_full, 4 * kHN * kBK * 2);
        for (int kb = 0; kb < 4; ++kb)
          tma_load_2d(smem + kHOffW + kb * (kHN * kBK * 2), &tmW1, w1_full, kb * kBK, ht * kHH);
        w1_issued = true;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
      bool ok = true;
      for (int kb = 0; kb < kNK; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&full[s], (kb / kStages) & 1, abort_flag, a.err) ||
            (I8 && !mbar_wait(&conv[s], (kb / kStages) & 1, abort_flag, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t aa = smem_u32(smem + S::kOffA + s * kATile), bb = smem_u32(smem + S::kOffB + s * kBTile);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc_mma(tbase, sdesc_sw128(aa + k * 32), sdesc_sw128(bb + k * 32), idesc, (kb | k) != 0);
        tc_commit(&empty[s]);
      }
      if (ok) tc_commit(acc_full);
    }
  } else {
    // ---- epilogue: experts, gates, this CTA's slice of r_t for both tasks
    const int q = warp & 3, grp = (warp - 2) >> 2;  // TMEM lane quarter; units [32 grp, 32 grp + 32) of the slice
    const int rl = q * 32 + lane, row = m0 + rl;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    // the biases and head constants, staged by the epilogue warps themselves while the first copies and MMAs run
    // (only these warps read them, all after this barrier)
    for (int k = threadIdx.x - 64; k < kBN; k += kEpiWarps * 32) {
      sbias[k] = __ldg(a.ple_b + n * kBN + k);
      if constexpr (I8) sscale[k] = __ldg(a.ple_s8 + n * kBN + k);
    }
    for (int k = threadIdx.x - 64; k < kHN; k += kEpiWarps * 32) {
      sb1[k] = __ldg(a.head_b1 + ht * kHH + k);
      sw2[k] = __ldg(a.head_w2 + ht * kHH + k);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    if constexpr (I8) {
      // 8-bit weights: stage s's [208][64] bytes -> the bf16 B tile in the layout a 128-byte-swizzled TMA load
      // would give (row r at 128 r, 16-byte chunk c at chunk c ^ (r % 8)); one 16-byte chunk of a row per step
      const int ct = threadIdx.x - 64;
      for (int kb = 0; kb < kNK; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait_warp(&wfull[s], (kb / kStages) & 1, abort_flag, a.err)) break;
        const uint8_t* src = smem + S::kOffW8 + s * kW8Tile;
        uint8_t* dst = smem + S::kOffB + s * kBTile;
        for (int c = ct; c < kBN * 4; c += kEpiWarps * 32) {
          const int r = c >> 2, kq = c & 3;
          uint4 lo, hi;
          s8x16_to_bf16(*reinterpret_cast<const uint4*>(src + r * 64 + kq * 16), lo, hi);
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, 2 * kq)) = lo;
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, 2 * kq + 1)) = hi;
        }
        fence_proxy_async_smem();  // the tile is read by the tensor cores (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[s]);
      }
    }
    const bool ok = mbar_wait_warp(acc_full, 0, abort_flag, a.err);
    if (ok) {
      tc_fence_after();
      uint32_t e[kNE][32], gl[16];
#pragma unroll
      for (int k = 0; k < kNE; ++k) tmem_ld32_nowait(tbase + lane_off + k * kSlice + grp * 32, e[k]);
      tmem_ld16_nowait(tbase + lane_off + kGateCol, gl);
      tmem_ld_wait();
      // per-task softmax over the 3 experts
      float g[kNT][kNE];
#pragma unroll
      for (int t = 0; t < kNT; ++t) {
        float l[kNE], mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kNE; ++k) {
          const int c = kGateCol + t * kNE + k;
          l[k] = (I8 ? __uint_as_float(gl[t * kNE + k]) * sscale[c] : __uint_as_float(gl[t * kNE + k])) + sbias[c];
          mx = fmaxf(mx, l[k]);
        }
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < kNE; ++k) {
          l[k] = expf(l[k] - mx);
          sum += l[k];
        }
        const float inv = 1.f / sum;
#pragma unroll
        for (int k = 0; k < kNE; ++k) g[t][k] = l[k] * inv;
      }
      // expert outputs ReLU(acc + b), kept in fp32 for r_t and staged (bf16) for the expert-output store
#pragma unroll
      for (int k = 0; k < kNE; ++k) {
        const float* bk = sbias + k * kSlice + grp * 32;
        const float* sk = sscale + k * kSlice + grp * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = I8 ? fmaf(__uint_as_float(e[k][j]), sk[j], bk[j]) : __uint_as_float(e[k][j]) + bk[j];
          e[k][j] = __float_as_uint(fmaxf(v, 0.f));
        }
        if (!a.keep_stages) continue;
        uint8_t* rowp = smem + S::kOffStage + (kNT + k) * kATile + rl * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(rowp + (((4 * grp + c) ^ (rl & 7)) << 4)) =
              make_uint4(pack_bf16(__uint_as_float(e[k][8 * c + 0]), __uint_as_float(e[k][8 * c + 1])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 2]), __uint_as_float(e[k][8 * c + 3])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 4]), __uint_as_float(e[k][8 * c + 5])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 6]), __uint_as_float(e[k][8 * c + 7])));
      }
      if (a.keep_stages && row < a.B && grp == 0 && n == 0) {
        float4* gd = reinterpret_cast<float4*>(a.gates + (int64_t)row * 8);
        gd[0] = make_float4(g[0][0], g[0][1], g[0][2], g[1][0]);
        gd[1] = make_float4(g[1][1], g[1][2], 0.f, 0.f);
      }
      // r_t for this thread's 32 units, staged as task t's slice
#pragma unroll
      for (int t = 0; t < kNT; ++t) {
        uint8_t* rowp = smem + S::kOffStage + t * kATile + rl * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t p[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int j = 8 * c + 2 * h;
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int k = 0; k < kNE; ++k) {
              x0 = fmaf(g[t][k], __uint_as_float(e[k][j]), x0);
              x1 = fmaf(g[t][k], __uint_as_float(e[k][j + 1]), x1);
            }
            p[h] = pack_bf16(x0, x1);
          }
          *reinterpret_cast<uint4*>(rowp + (((4 * grp + c) ^ (rl & 7)) << 4)) = make_uint4(p[0], p[1], p[2], p[3]);
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();  // the staged tiles are read by TMA stores (async proxy)
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    if (threadIdx.x == 64) {
      if (ok) {
        // r_t slices first (the heads wait for them), the expert outputs (when kept) in a second group
        for (int t = 0; t < kNT; ++t) tma_store_2d(&tmR, smem + S::kOffStage + t * kATile, n * kSlice, t * r_rows + m0);
        bulk_commit();
        if (a.keep_stages)
          for (int k = 0; k < kNE; ++k)
            tma_store_2d(&tmEx, smem + S::kOffStage + (kNT + k) * kATile, k * kDE + n * kSlice, m0);
        bulk_commit();
        asm volatile("cp.async.bulk.wait_group 1;" ::: "memory");  // the r_t slices are written
        bulk_wait_read<0>();  // and the staging area has been read (the head operands reuse it)
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }
  // ---- heads: every slice of the row block's R is written once all four CTAs of the cluster are here
  cluster_sync();
  if (warp == 0 && lane == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");  // R is read by TMA, as it was written
    mbar_expect_tx(h_full, w1_early ? 4 * kATile : kHBytes);
    for (int kb = 0; kb < 4; ++kb) {
      tma_load_2d(smem + kb * kATile, &tmR, h_full, kb * kBK, ht * r_rows + m0);
      if (!w1_early) tma_load_2d(smem + kHOffW + kb * (kHN * kBK * 2), &tmW1, h_full, kb * kBK, ht * kHH);
    }
    if (w1_early && !w1_issued) mbar_arrive(w1_full);  // (gave up before issuing them: nothing will land)
    // the error bits of every earlier kernel of the call (complete once the wait returns) and of this CTA's own
    // waits so far, read while the head MMAs run
    pdl_wait();
    err_seen = *reinterpret_cast<volatile int*>(a.err);
  } else if (warp == 1 && lane == 0) {
    if (mbar_wait(h_full, 0, abort_flag, a.err) && (!w1_early || mbar_wait(w1_full, 0, abort_flag, a.err))) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(kBM, kHN);
      for (int kb = 0; kb < 4; ++kb)
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc_mma(tbase, sdesc_sw128(smem_u32(smem + kb * kATile) + k * 32),
                 sdesc_sw128(smem_u32(smem + kHOffW + kb * (kHN * kBK * 2)) + k * 32), idesc, (kb | k) != 0);
      tc_commit(head_full);
    } else {
      mbar_drain(h_full, 0);  // (gave up: the loads land before the shared memory is released)
      if (w1_early) mbar_drain(w1_full, 0);
    }
  }
  if (warp >= 2) {
    // ReLU(h + b1) . w2: warp group grp sums hidden units [64 grp, 64 grp + 64) of each row; the two partial logits
    // meet in shared memory, and the rows [64 hh, 64 hh + 64) of this CTA's half are finished (bias, sigmoid)
    const int q = warp & 3, grp = (warp - 2) >> 2, rl = q * 32 + lane;
    float part = 0.f;
    if (mbar_wait_warp(head_full, 0, abort_flag, a.err)) {
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16) + grp * 64, v);
      tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16) + grp * 64 + 32, v + 32);
      tmem_ld_wait();
      const float* b1 = sb1 + grp * 64;
      const float* w2 = sw2 + grp * 64;
#pragma unroll
      for (int j = 0; j < 64; ++j) part = fmaf(fmaxf(__uint_as_float(v[j]) + b1[j], 0.f), w2[j], part);
    }
    plog[grp * kBM + rl] = part;
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    const int row = m0 + rl;
    if (grp == 0 && (rl >> 6) == hh) {
      const float logit = (plog[rl] + plog[kBM + rl]) + a.head_b2[ht];
      if (row < a.B) a.out[(int64_t)row * kNT + ht] = 1.f / (1.f + expf(-logit));
    }
  }
  if (threadIdx.x == 64) bulk_wait_read<0>();  // (the stores' shared-memory source is read before the CTA exits)
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  // This is the last kernel of a call. Each CTA ORs what it read of the error word, and a timeout of its own later
  // waits (they raise the CTA's abort flag), into the pinned host word, which the host reads after waiting for the
  // stream. An error-free call ends without an atomic or a round trip to host memory. The device word keeps its
  // bits until the host, having found an error, clears it.
  if (threadIdx.x == 0) {
    const int ew = err_seen | (*abort_flag ? kErrTimeout : 0);
    if (ew) atomicOr(a.err_host, ew);
  }
}

}  // namespace

cudaError_t prepare_ple_kernel() {
  cudaError_t e = cudaFuncSetAttribute(ple_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<false>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ple_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<true>::kBytes);
  return e;
}

cudaError_t launch_ple_heads(const FwdArgs& a, const CUtensorMap& tmY, const CUtensorMap& tmW, const CUtensorMap& tmR,
                             const CUtensorMap& tmEx, const CUtensorMap& tmW1, int r_rows, cudaStream_t s) {
  const int blocks = (a.B + kBM - 1) / kBM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks * kSlices);
  cfg.blockDim = dim3(kThreads);
  const bool i8 = a.ple_s8 != nullptr;
  cfg.dynamicSmemBytes = i8 ? Smem<true>::kBytes : Smem<false>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the four CTAs of a row block
  attr[0].val.clusterDim.x = kSlices;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  return i8 ? cudaLaunchKernelEx(&cfg, ple_kernel<true>, a, tmY, tmW, tmR, tmEx, tmW1, r_rows)
            : cudaLaunchKernelEx(&cfg, ple_kernel<false>, a, tmY, tmW, tmR, tmEx, tmW1, r_rows);
}

}  // namespace cvr
