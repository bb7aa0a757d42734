// PLE experts, task gates and prediction heads of the CVR forward pass (iQIYI ad-CVR article, section 3.2.4:
// three single-layer experts over the flattened tokens, a softmax gate per task, and per task a two-layer head
// ending in a sigmoid pCVR).
//
//  ple_kernel    four CTAs per 128-row block. CTA n computes, for the block's rows, the 208 columns
//                  [e_0 units 64n..64n+63 | e_1 units .. | e_2 units .. | the 6 gate logits | 10 zero columns]
//                of Y . W^T (Y [rows][2048] bf16, K = 2048) on tcgen05 with the accumulator in TMEM, A and B
//                streamed by TMA through a 5-stage mbarrier ring. Every CTA has all gate logits, so each forms
//                its 64-unit slice of r_t = sum_k g_t[k] ReLU(e_k + b_k) for both tasks (fp32, then bf16) and
//                writes it with TMA stores into R [task][row][256], next to the expert outputs and the gates;
//                then it counts its row block as done.
//  heads         the four CTAs of a row block form a cluster. Once all four slices of R are written (one cluster
//                barrier), CTA n computes hidden units [64 (n % 2), +64) of task n / 2's head, ReLU(W1_t r_t +
//                b1) on tcgen05 (M=128, N=64, K=256) with r_t read back through L2 and its W1 rows loaded into the
//                ring, applies its half of the 128 -> 1 layer and sends the partial logits to the task's first
//                CTA over distributed shared memory, which adds the two halves in order, the bias and the sigmoid.
//
// The kernel starts per row block instead of waiting for the whole Token Mixer grid: a CTA waits (bounded)
// until the Token Mixer has counted every tile of its row block as written, so the first blocks run on the SMs
// the Token Mixer's last round leaves free. The counters are cleared by the first kernel of every call.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kSlice = 64;                  // units of each expert per CTA
constexpr int kSlices = kDE / kSlice;       // 4 CTAs per 128-row block
constexpr int kBN = kNE * kSlice + 16;      // 208 columns per CTA: 3 x 64 expert units + 16 gate columns
constexpr int kGateCol = kNE * kSlice;      // 192: the 6 gate logits (task-major), then zero columns
constexpr int kBM = 128, kBK = 64, kStages = 5;
constexpr int kATile = kBM * kBK * 2;       // 16 KB
constexpr int kBTile = kBN * kBK * 2;       // 26 KB
constexpr int kNK = kYD / kBK;              // 32 k-blocks
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..9 epilogue
constexpr int kTmemCols = 256;
static_assert(kPleCols == kSlices * kBN, "four 208-column slices");

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kStages * kATile;
constexpr int kRingBytes = kStages * (kATile + kBTile);   // 210 KB
// output staging, in the ring once the main loop is done: r_t slices [task] then expert slices [k], each
// [128 rows][64 units] bf16 with the 128-byte swizzle (the layout of a TMA box of 64 x 128)
constexpr int kOffStage = 0;
static_assert((kNT + kNE) * kATile <= kRingBytes, "output staging fits the ring");
// heads, in the ring as well: r_t (4 K-blocks of [128][64]) then this CTA's W1 rows (4 K-blocks of [64][64])
constexpr int kHN = kHH / 2;                // hidden units per CTA
constexpr int kHOffW = 4 * kATile;
constexpr int kHBytes = 4 * kATile + 4 * kHN * kBK * 2;  // 96 KB
static_assert(kHBytes <= kRingBytes, "head operands fit the ring");
constexpr int kOffBias = kRingBytes;                      // fp32 slice bias [208], head b1 / w2 of this half [64] each
constexpr int kOffPlog = kOffBias + (kBN + 2 * kHN) * 4;  // fp32 [2 halves][128 rows]: partial logits (task's first CTA)
constexpr int kOffBar = kOffPlog + 2 * kBM * 4;
constexpr int kNBar = 2 * kStages + 1 + 2;
constexpr int kSmemBytes = kOffBar + kNBar * 8 + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// every thread of every CTA of the cluster arrives; memory before it (shared and global) is visible after it
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}
// Waits (at most ~1 s) until *cnt >= need; a wait that gives up is reported and the kernel goes on (every access
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

__global__ void __launch_bounds__(kThreads, 1)
    ple_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmY,
               const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmR,
               const __grid_constant__ CUtensorMap tmEx, const __grid_constant__ CUtensorMap tmW1, int r_rows) {
  extern __shared__ uint8_t smem_raw[];
  CVR_TL_BEGIN(TL_PLE_HEADS);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sbias = reinterpret_cast<float*>(smem + kOffBias);  // [208]
  float* sb1 = sbias + kBN;                                  // [64]
  float* sw2 = sb1 + kHN;                                    // [64]
  float* plog = reinterpret_cast<float*>(smem + kOffPlog);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bar;
  uint64_t* empty = bar + kStages;
  uint64_t* acc_full = bar + 2 * kStages;  // the main loop's accumulator is complete
  uint64_t* h_full = acc_full + 1;         // heads: r_t and the W1 rows landed
  uint64_t* head_full = acc_full + 2;      // heads: hidden pre-activations complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = (int)blockIdx.x % kSlices;            // slice of this CTA (= its rank in the cluster)
  const int rb = (int)blockIdx.x / kSlices;           // row block
  const int m0 = rb * kBM;
  const int ht = n >> 1, hh = n & 1;                  // head task and hidden half of this CTA
  for (int k = threadIdx.x; k < kBN; k += blockDim.x) sbias[k] = __ldg(a.ple_b + n * kBN + k);  // (constants)
  for (int k = threadIdx.x; k < kHN; k += blockDim.x) {
    sb1[k] = __ldg(a.head_b1 + ht * kHH + hh * kHN + k);
    sw2[k] = __ldg(a.head_w2 + ht * kHH + hh * kHN + k);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(h_full, 1);
    mbar_init(head_full, 1);
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // weights first: they do not depend on the Token Mixer
      const int pre = kStages < kNK ? kStages : kNK;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_expect_tx(&full[kb], kATile + kBTile);
        tma_load_2d(smem + kOffB + kb * kBTile, &tmW, &full[kb], kb * kBK, n * kBN);
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
          mbar_expect_tx(&full[s], kATile + kBTile);
          tma_load_2d(smem + kOffB + s * kBTile, &tmW, &full[s], kb * kBK, n * kBN);
        }
        tma_load_2d(smem + kOffA + s * kATile, &tmY, &full[s], kb * kBK, m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
      bool ok = true;
      for (int kb = 0; kb < kNK; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&full[s], (kb / kStages) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t aa = smem_u32(smem + kOffA + s * kATile), bb = smem_u32(smem + kOffB + s * kBTile);
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
          l[k] = __uint_as_float(gl[t * kNE + k]) + sbias[kGateCol + t * kNE + k];
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
#pragma unroll
        for (int j = 0; j < 32; ++j) e[k][j] = __float_as_uint(fmaxf(__uint_as_float(e[k][j]) + bk[j], 0.f));
        uint8_t* rowp = smem + kOffStage + (kNT + k) * kATile + rl * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(rowp + (((4 * grp + c) ^ (rl & 7)) << 4)) =
              make_uint4(pack_bf16(__uint_as_float(e[k][8 * c + 0]), __uint_as_float(e[k][8 * c + 1])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 2]), __uint_as_float(e[k][8 * c + 3])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 4]), __uint_as_float(e[k][8 * c + 5])),
                         pack_bf16(__uint_as_float(e[k][8 * c + 6]), __uint_as_float(e[k][8 * c + 7])));
      }
      if (row < a.B && grp == 0 && n == 0) {
        float4* gd = reinterpret_cast<float4*>(a.gates + (int64_t)row * 8);
        gd[0] = make_float4(g[0][0], g[0][1], g[0][2], g[1][0]);
        gd[1] = make_float4(g[1][1], g[1][2], 0.f, 0.f);
      }
      // r_t for this thread's 32 units, staged as task t's slice
#pragma unroll
      for (int t = 0; t < kNT; ++t) {
        uint8_t* rowp = smem + kOffStage + t * kATile + rl * 128;
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
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    if (threadIdx.x == 64) {
      if (ok) {
        // r_t slices first (the heads wait for them), the expert outputs in a second group
        for (int t = 0; t < kNT; ++t) tma_store_2d(&tmR, smem + kOffStage + t * kATile, n * kSlice, t * r_rows + m0);
        bulk_commit();
        for (int k = 0; k < kNE; ++k)
          tma_store_2d(&tmEx, smem + kOffStage + (kNT + k) * kATile, k * kDE + n * kSlice, m0);
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
    mbar_expect_tx(h_full, kHBytes);
    for (int kb = 0; kb < 4; ++kb) {
      tma_load_2d(smem + kb * kATile, &tmR, h_full, kb * kBK, ht * r_rows + m0);
      tma_load_2d(smem + kHOffW + kb * (kHN * kBK * 2), &tmW1, h_full, kb * kBK, ht * kHH + hh * kHN);
    }
  } else if (warp == 1 && lane == 0) {
    if (mbar_wait(h_full, 0, abort_flag, a.err)) {
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
    }
  }
  if (warp >= 2 && warp < 6) {
    // ReLU(h + b1) . w2 over this CTA's 64 hidden units: the partial logit of each row goes to the task's first CTA
    const int q = warp & 3, rl = q * 32 + lane;
    float part = 0.f;
    if (mbar_wait_warp(head_full, 0, abort_flag, a.err)) {
      tc_fence_after();
      uint32_t v[kHN];
      tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16), v);
      tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16) + 32, v + 32);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < kHN; ++j) part = fmaf(fmaxf(__uint_as_float(v[j]) + sb1[j], 0.f), sw2[j], part);
    }
    st_cluster_f32(peer_addr(smem_u32(plog + hh * kBM + rl), (uint32_t)(2 * ht)), part);
  }
  cluster_sync();
  if (hh == 0 && warp >= 2 && warp < 6) {
    const int q = warp & 3, rl = q * 32 + lane, row = m0 + rl;
    const float logit = (plog[rl] + plog[kBM + rl]) + a.head_b2[ht];
    if (row < a.B) a.out[(int64_t)row * kNT + ht] = 1.f / (1.f + expf(-logit));
  }
  if (threadIdx.x == 64) bulk_wait_all();  // (the expert outputs are written before the CTA exits)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  // This is the last kernel of a call: the last of its CTAs to finish moves the call's error bits (once every
  // earlier kernel has completed) into the host word and resets the device word for the next call. The host word
  // is touched only when there is an error (the host reads it after waiting for the stream, which makes the write
  // visible), so an error-free call ends without a round trip to host memory.
  if (threadIdx.x == 0) {
    pdl_wait();
    __threadfence();
    if (atomicAdd(a.done, 1u) == gridDim.x - 1) {
      __threadfence();
      const int ew = atomicExch(a.err, 0);
      if (ew) {
        volatile int* hw = a.err_host;
        *hw = *hw | ew;
      }
      atomicExch(a.done, 0u);
    }
  }
}

}  // namespace

cudaError_t prepare_ple_kernel() {
  return cudaFuncSetAttribute(ple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_ple_heads(const FwdArgs& a, const CUtensorMap& tmY, const CUtensorMap& tmW, const CUtensorMap& tmR,
                             const CUtensorMap& tmEx, const CUtensorMap& tmW1, int r_rows, cudaStream_t s) {
  const int blocks = (a.B + kBM - 1) / kBM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks * kSlices);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, ple_kernel, a, tmY, tmW, tmR, tmEx, tmW1, r_rows);
}

}  // namespace cvr
