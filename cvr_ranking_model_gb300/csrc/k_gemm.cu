// tcgen05 GEMMs of the CVR forward pass with fused epilogues, and the prediction heads.
//
//  gemm_kernel<EPI>  D[128 x BN] = A[128 x K] . W[BN x K]^T, both operands bf16 K-major in 128B-swizzled
//                    shared memory loaded by TMA through a STAGES-deep mbarrier ring; one elected thread
//                    issues tcgen05.mma into a TMEM accumulator; four epilogue warps drain TMEM with
//                    tcgen05.ld (one accumulator row per thread) and apply:
//    EPI_TOKENIZE    [Z[:, 0:1664] | Q] = bf16(I . [Wtok_item ; Wq_x Wtok_item]^T + [xu | qu + qb][request])
//                    (iQIYI 3.2.2 and 3.2.3 item 1): the tokens and, since the first layer's query FFN is
//                    linear in them, that layer's queries, with the query weights folded into the tokeniser
//                    (Wq_x Wtok precomputed); the per-request terms -- user half of the tokeniser and of
//                    the folded query, biases, mean-pool term qb -- are computed once per request
//                    (iQIYI 3.4.5)
//    EPI_QUERY       Q = bf16(flat(X) . Wq_x^T + qb[request]) for stacked layers (iQIYI 3.2.3, item 1)
//    EPI_PLE         Ex = bf16(ReLU(Y . We^T + be)); the 6 gate logits of the last tile become per-task
//                    softmax weights over the 3 experts                          (iQIYI 3.2.4)
//  heads_kernel      per task t: r_t = sum_k gate_t[k] e_k built in shared memory, ReLU(W1_t r_t + b1)
//                    on tcgen05, then the 128 -> 1 output and sigmoid in the epilogue (iQIYI 3.2.4).
#include "cvr_internal.cuh"

namespace cvr {

namespace {

enum { EPI_TOKENIZE = 0, EPI_QUERY = 1, EPI_PLE = 2 };
constexpr int kThreads = 576;  // heads kernel: warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..17 build r_t,
                               // warps 2..5 then drain TMEM (one per lane quarter)
constexpr int kBuildWarps = kThreads / 32 - 2;
constexpr int kBM = 128, kBK = 64;
constexpr int kATile = kBM * kBK * 2;  // 16 KB

// named barrier of the NEPI epilogue warps (the producer and MMA warps never take part)
template <int NEPI>
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NEPI * 32) : "memory");
}

template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
  return BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
}
template <int BN, int STAGES, int EPI>
__host__ __device__ constexpr int gemm_smem_bytes() {
  return 1024 + STAGES * (kATile + BN * kBK * 2) + 256 + (kPleCols + 32) * 4 +  // + PLE biases
         (EPI == EPI_TOKENIZE ? 1024 + 2 * kBM * BN * 2                               // + output staging (aligned):
                              : EPI == EPI_PLE ? 1024 + kBM * BN * 2 : 0);            //   two swizzled tiles / one plain
}

// Persistent GEMM: CTAs loop over 128 x BN output tiles (n fastest, so co-running CTAs share A rows in L2).
// Warp 0 streams A/B k-blocks through a STAGES-deep ring; warp 1 issues the MMAs into one of two TMEM
// accumulators; NEPI epilogue warps drain the other one, so a tile's epilogue overlaps the next tile's
// MMAs. With 8 epilogue warps the two warpgroups split the 32-column chunks of a tile.
template <int BN, int STAGES, int EPI, int NEPI>
__global__ void __launch_bounds__(64 + NEPI * 32, 1)
    gemm_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmZo,
                const __grid_constant__ CUtensorMap tmQo, int M, int N, int K, int layer) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int B_TILE = BN * kBK * 2;
  constexpr uint32_t TC = tmem_cols<BN>();
  constexpr int NCHUNK = (BN + 31) / 32;
  constexpr int NGRP = NEPI / 4;
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kATile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_TILE);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* sbias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 256);  // PLE: biases of all columns
  // output staging for TMA stores (1024-byte aligned): tokeniser, two tiles [128][BN] bf16 as boxes of [128 rows]
  // [64 columns] with the 128-byte swizzle; PLE, one plain [128][BN] tile
  uint8_t* sOut = reinterpret_cast<uint8_t*>(((reinterpret_cast<uintptr_t>(sbias + kPleCols + 32)) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (EPI == EPI_PLE)  // constant: staged before waiting for the previous kernel
    for (int k = threadIdx.x; k < kPleCols + 32; k += blockDim.x) sbias[k] = __ldg(a.ple_b + k);
  const int tiles_n = N / BN;
  const int n_tiles = ((M + kBM - 1) / kBM) * tiles_n;
  const int nk = K / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], NEPI);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tslot, 2 * TC);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      int kc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / tiles_n) * kBM, n0 = (tile % tiles_n) * BN;
        for (int kb = 0; kb < nk; ++kb, ++kc) {
          const int s = kc % STAGES;
          if (kc >= STAGES && !mbar_wait(&empty[s], ((kc / STAGES) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], kATile + B_TILE);
          tma_load_2d(sA + s * kATile, &tmA, &full[s], kb * kBK, m0);
          tma_load_2d(sB + s * B_TILE, &tmB, &full[s], kb * kBK, n0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, BN);
      int kc = 0, i = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait(&acc_empty[buf], ((i >> 1) & 1) ^ 1, abort_flag, a.err)) break;
        const uint32_t dacc = tbase + buf * TC;
        for (int kb = 0; kb < nk; ++kb, ++kc) {
          const int s = kc % STAGES;
          if (!mbar_wait(&full[s], (kc / STAGES) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aa = smem_u32(sA + s * kATile), bb = smem_u32(sB + s * B_TILE);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma(dacc, sdesc_sw128(aa + k * 32), sdesc_sw128(bb + k * 32), idesc, (kb | k) != 0);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&acc_full[buf]);
      }
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;     // chunk group
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int i = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
      const int m0 = (tile / tiles_n) * kBM, n0 = (tile % tiles_n) * BN;
      const int buf = i & 1;
      const int row = m0 + q * 32 + lane;
      const bool live = row < M;
      int req = 0;
      if (EPI != EPI_PLE && live) req = min(max(a.req_ids[row], 0), a.R - 1);
      // the addends of this warp's chunks (per-request terms or biases) are loaded before waiting for the
      // accumulator, so their latency hides under the tile's MMAs
      constexpr int NMY = (NCHUNK + NGRP - 1) / NGRP;
      float addv[NMY][32];
#pragma unroll
      for (int m = 0; m < NMY; ++m) {
        const int c = grp + m * NGRP, nb = n0 + c * 32;
        if (c >= NCHUNK || !live) continue;
        if (EPI == EPI_TOKENIZE) {
          ldg32(a.xu + (int64_t)req * kTokN + nb, addv[m]);
          if (nb >= kXD && !a.q_add) {  // first-layer query columns: + the mean-pool term of the request
            float qadd[32];
            ldg32(a.qb + (int64_t)req * (kG * kD) + (nb - kXD), qadd);
#pragma unroll
            for (int x = 0; x < 32; ++x) addv[m][x] += qadd[x];
          }
        } else if (EPI == EPI_QUERY) {
          ldg32(a.qb + ((int64_t)layer * a.R + req) * (kG * kD) + nb, addv[m]);
        }
      }
      if (!mbar_wait(&acc_full[buf], (i >> 1) & 1, abort_flag, a.err)) break;
      tc_fence_after();
      uint8_t* sb = sOut + (EPI == EPI_TOKENIZE ? (i & 1) * (kBM * BN * 2) : 0);
      if (EPI == EPI_TOKENIZE || (EPI == EPI_PLE && i > 0)) {
        // the TMA store issued from this staging buffer earlier must have finished reading it
        if (threadIdx.x == 64) {
          if (EPI == EPI_TOKENIZE)
            bulk_wait_read<1>();
          else
            bulk_wait_read<0>();
        }
        epi_bar<NEPI>();
      }
#pragma unroll
      for (int m = 0; m < NMY; ++m) {
        const int c = grp + m * NGRP;
        if (c >= NCHUNK) continue;
        float v[32];
        const float* add = EPI == EPI_PLE ? sbias + n0 + c * 32 : addv[m];
        const int nb = n0 + c * 32;
        tmem_ld32(tbase + lane_off + buf * TC + c * 32, v);
        if (!live) continue;
        if (EPI == EPI_TOKENIZE) {
          // columns [32c, 32c + 32) of row rl into the staging tile: box c/2, 16-byte chunks 4 (c%2) + j, swizzled
          const int rl = q * 32 + lane;
          uint8_t* rowp = sb + (c >> 1) * (kBM * 128) + rl * 128;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 p;
            p.x = pack_bf16(v[8 * j + 0] + add[8 * j + 0], v[8 * j + 1] + add[8 * j + 1]);
            p.y = pack_bf16(v[8 * j + 2] + add[8 * j + 2], v[8 * j + 3] + add[8 * j + 3]);
            p.z = pack_bf16(v[8 * j + 4] + add[8 * j + 4], v[8 * j + 5] + add[8 * j + 5]);
            p.w = pack_bf16(v[8 * j + 6] + add[8 * j + 6], v[8 * j + 7] + add[8 * j + 7]);
            *reinterpret_cast<uint4*>(rowp + ((((c & 1) * 4 + j) ^ (rl & 7)) << 4)) = p;
          }
        } else if (EPI == EPI_QUERY) {
          __nv_bfloat16* out = a.Q + (int64_t)row * (kG * kD) + nb;
          uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (c * 32 + j * 8 >= BN) break;
            uint4 p;
            p.x = pack_bf16(v[8 * j + 0] + add[8 * j + 0], v[8 * j + 1] + add[8 * j + 1]);
            p.y = pack_bf16(v[8 * j + 2] + add[8 * j + 2], v[8 * j + 3] + add[8 * j + 3]);
            p.z = pack_bf16(v[8 * j + 4] + add[8 * j + 4], v[8 * j + 5] + add[8 * j + 5]);
            p.w = pack_bf16(v[8 * j + 6] + add[8 * j + 6], v[8 * j + 7] + add[8 * j + 7]);
            dst[j] = p;
          }
        } else {  // EPI_PLE
          // ReLU(expert) columns of row rl into the plain [128][BN] staging tile (the TMA store clips the
          // columns past the 768 expert outputs)
          const int rl = q * 32 + lane;
          uint4* rowp = reinterpret_cast<uint4*>(sb + rl * (BN * 2) + c * 64);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (c * 32 + j * 8 >= BN) break;
            uint4 p;
            uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              pp[e] = pack_bf16(fmaxf(v[8 * j + 2 * e] + add[8 * j + 2 * e], 0.f),
                                fmaxf(v[8 * j + 2 * e + 1] + add[8 * j + 2 * e + 1], 0.f));
            rowp[j] = p;
          }
          // gate logits sit in columns [768, 774): 16 columns into the chunk that starts at 752 (tiles of
          // 208 start at 624, chunks every 32 columns), a compile-time offset so v and add stay in registers
          constexpr int o = 16;
          static_assert(EPI != EPI_PLE || ((kPleN - o) % BN) % 32 == 0, "gate logits 16 columns into a chunk");
          if (nb + o == kPleN) {
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
              float l0 = v[o + 3 * t] + add[o + 3 * t];
              float l1 = v[o + 3 * t + 1] + add[o + 3 * t + 1];
              float l2 = v[o + 3 * t + 2] + add[o + 3 * t + 2];
              const float mx = fmaxf(l0, fmaxf(l1, l2));
              l0 = expf(l0 - mx);
              l1 = expf(l1 - mx);
              l2 = expf(l2 - mx);
              const float inv = 1.f / (l0 + l1 + l2);
              float* gd = a.gates + (int64_t)row * 8 + 3 * t;
              gd[0] = l0 * inv;
              gd[1] = l1 * inv;
              gd[2] = l2 * inv;
            }
          }
        }
      }
      if (EPI == EPI_TOKENIZE || EPI == EPI_PLE) {
        // the whole tile is staged: one thread stores it (tokeniser: boxes of 64 columns, tokens into Z and the
        // first layer's queries into Q; PLE: one box of BN columns into the expert outputs)
        fence_proxy_async_smem();
        epi_bar<NEPI>();
        if (threadIdx.x == 64) {
          if (EPI == EPI_TOKENIZE) {
            const bool qcols = n0 >= kXD;
#pragma unroll
            for (int bx = 0; bx < BN / 64; ++bx)
              tma_store_2d(qcols ? &tmQo : &tmZo, sb + bx * (kBM * 128), (qcols ? n0 - kXD : n0) + bx * 64, m0);
          } else {
            tma_store_2d(&tmZo, sb, n0, m0);
          }
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if ((EPI == EPI_TOKENIZE || EPI == EPI_PLE) && threadIdx.x == 64) bulk_wait_all();  // stores landed before exit
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * TC);
  }
}

// ------------------------------------------------------------------------------------------
// prediction heads: grid (ceil(B/128), tasks)
constexpr int kHeadSmem = 1024 + 4 * kATile + 4 * kATile + 256 + 2 * kHH * 4;

__global__ void __launch_bounds__(kThreads, 1) heads_kernel(const __grid_constant__ FwdArgs a,
                                                            const __grid_constant__ CUtensorMap tmW1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                 // r_t tile: 4 K-blocks of [128][64] bf16, 128B-swizzled
  uint8_t* sW = smem + 4 * kATile;    // W1_t: 4 K-blocks of [128][64]
  uint64_t* barA = reinterpret_cast<uint64_t*>(sW + 4 * kATile);
  uint64_t* barW = barA + 1;
  uint64_t* barD = barW + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(barD + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* sB1 = reinterpret_cast<float*>(sW + 4 * kATile + 256);  // b1_t, then w2_t: constants, loaded up front
  float* sW2 = sB1 + kHH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, t = blockIdx.y;
  if (threadIdx.x < kHH) {  // (weights: no dependency on the previous kernel)
    sB1[threadIdx.x] = __ldg(a.head_b1 + t * kHH + threadIdx.x);
    sW2[threadIdx.x] = __ldg(a.head_w2 + t * kHH + threadIdx.x);
  }
  if (threadIdx.x == 0) {
    mbar_init(barA, kBuildWarps * 32);
    mbar_init(barW, 1);
    mbar_init(barD, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();
  if (warp == 0 && lane == 0) {  // W1_t is constant: its load overlaps the previous kernel
    mbar_expect_tx(barW, 4 * kATile);
    for (int kb = 0; kb < 4; ++kb) tma_load_2d(sW + kb * kATile, &tmW1, barW, kb * kBK, t * kHH);
  }
  pdl_wait();
  if (warp == 0) {
  } else if (warp == 1) {
    if (lane == 0) {
      if (mbar_wait(barA, 0, abort_flag, a.err) && mbar_wait(barW, 0, abort_flag, a.err)) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16(kBM, kHH);
        for (int kb = 0; kb < 4; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma(tbase, sdesc_sw128(smem_u32(sA + kb * kATile) + k * 32), sdesc_sw128(smem_u32(sW + kb * kATile) + k * 32),
                   idesc, (kb | k) != 0);
        tc_commit(barD);
      }
    }
  } else {
    const int q = warp & 3;
    const int rl = q * 32 + lane;
    const int row = m0 + rl;
    const bool live = row < a.B;
    // r_t = sum_k gate_t[k] e_k for the tile's 128 rows: build warp w builds rows w, w + 16, ...; lane l
    // covers hidden units [8l, 8l+8) (a 16-byte vector of each expert), four rows' loads in flight at once.
    const int ew = warp - 2;
#pragma unroll 1
    for (int r0 = ew; r0 < kBM; r0 += 4 * kBuildWarps) {
      uint4 u[4][3];
      float g[4][3];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = r0 + kBuildWarps * k, grow = m0 + rr;
        const bool ok = grow < a.B;
        const uint4* e = reinterpret_cast<const uint4*>(a.Ex + (int64_t)(ok ? grow : 0) * kPleN);
#pragma unroll
        for (int x = 0; x < 3; ++x) {
          u[k][x] = ok ? __ldg(e + x * (kDE / 8) + lane) : make_uint4(0, 0, 0, 0);
          g[k][x] = ok ? __ldg(a.gates + (int64_t)grow * 8 + 3 * t + x) : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = r0 + kBuildWarps * k;
        const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u[k][0]);
        const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u[k][1]);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u[k][2]);
        uint4 p;
        uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = g[k][0] * __low2float(h0[i]) + g[k][1] * __low2float(h1[i]) + g[k][2] * __low2float(h2[i]);
          const float x1 = g[k][0] * __high2float(h0[i]) + g[k][1] * __high2float(h1[i]) + g[k][2] * __high2float(h2[i]);
          pp[i] = pack_bf16(x0, x1);
        }
        *reinterpret_cast<uint4*>(sA + (lane >> 3) * kATile + sw128_offset(rr, lane & 7)) = p;
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(barA);
    if (warp < 6 && mbar_wait(barD, 0, abort_flag, a.err)) {
      tc_fence_after();
      float logit = 0.f;
#pragma unroll 1
      for (int c = 0; c < kHH / 32; c += 2) {  // two TMEM loads in flight, b1 and w2 from shared memory
        uint32_t v[64];
        tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16) + c * 32, v);
        tmem_ld32_nowait(tbase + ((uint32_t)(q * 32) << 16) + c * 32 + 32, v + 32);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 64; ++j) logit += fmaxf(__uint_as_float(v[j]) + sB1[c * 32 + j], 0.f) * sW2[c * 32 + j];
      }
      if (live) a.out[(int64_t)row * kNT + t] = 1.f / (1.f + expf(-(logit + a.head_b2[t])));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
  // This is the last kernel of a call: every earlier kernel has completed (programmatic dependencies chain),
  // so the last of its CTAs to finish publishes the call's error bits to the host word and resets the
  // device word for the next call.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.done, 1u) == gridDim.x * gridDim.y - 1) {
      __threadfence();
      const int e = atomicExch(a.err, 0);
      volatile int* hw = a.err_host;
      *hw = *hw | e;
      atomicExch(a.done, 0u);
      __threadfence_system();
    }
  }
}

template <int BN, int STAGES, int EPI, int NEPI>
cudaError_t prepare_gemm() {
  return cudaFuncSetAttribute(gemm_kernel<BN, STAGES, EPI, NEPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              gemm_smem_bytes<BN, STAGES, EPI>());
}

// a persistent grid of at most max_grid CTAs (0: one per SM)
template <int BN, int STAGES, int EPI, int NEPI>
cudaError_t launch_gemm(const FwdArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmZo,
                        const CUtensorMap& tmQo, int M, int N, int K, int layer, cudaStream_t s, int max_grid = 0) {
  const int tiles = ((M + kBM - 1) / kBM) * (N / BN);
  const int cap = max_grid > 0 && max_grid < a.num_sms ? max_grid : a.num_sms;
  const int grid = tiles < cap ? tiles : cap;
  return launch_kernel(gemm_kernel<BN, STAGES, EPI, NEPI>, dim3(grid), dim3(64 + NEPI * 32), gemm_smem_bytes<BN, STAGES, EPI>(),
                       s, a.pdl != 0, a, tmA, tmB, tmZo, tmQo, M, N, K, layer);
}

constexpr int kTokBN = 128, kTokStages = 4, kTokEpi = 8;
constexpr int kQryBN = 96, kQryStages = 6, kQryEpi = 8;
constexpr int kPleBN = 208, kPleStages = 4, kPleEpi = 8;
static_assert(kPleCols % kPleBN == 0, "PLE columns are a whole number of tiles");

}  // namespace

cudaError_t prepare_gemm_kernels() {
  cudaError_t e = prepare_gemm<kTokBN, kTokStages, EPI_TOKENIZE, kTokEpi>();
  if (e == cudaSuccess) e = prepare_gemm<kQryBN, kQryStages, EPI_QUERY, kQryEpi>();
  if (e == cudaSuccess) e = prepare_gemm<kPleBN, kPleStages, EPI_PLE, kPleEpi>();
  if (e == cudaSuccess) e = cudaFuncSetAttribute(heads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHeadSmem);
  return e;
}

cudaError_t launch_tokenizer(const FwdArgs& a, const CUtensorMap& tmI, const CUtensorMap& tmW, const CUtensorMap& tmZo,
                             const CUtensorMap& tmQo, int max_grid, cudaStream_t s) {
  static_assert(kXD % kTokBN == 0 && kTokN % kTokBN == 0, "token and query columns fall in separate tiles");
  static_assert(kTokBN % 64 == 0 && gemm_smem_bytes<kTokBN, kTokStages, EPI_TOKENIZE>() <= 232448, "staging fits");
  return launch_gemm<kTokBN, kTokStages, EPI_TOKENIZE, kTokEpi>(a, tmI, tmW, tmZo, tmQo, a.B, kTokN, kID, 0, s, max_grid);
}

cudaError_t launch_query(const FwdArgs& a, int layer, const CUtensorMap& tmX, const CUtensorMap& tmW, cudaStream_t s) {
  return launch_gemm<kQryBN, kQryStages, EPI_QUERY, kQryEpi>(a, tmX, tmW, tmX, tmX, a.B, kG * kD, kXD, layer, s);
}

cudaError_t launch_ple(const FwdArgs& a, const CUtensorMap& tmY, const CUtensorMap& tmW, const CUtensorMap& tmEx,
                       cudaStream_t s) {
  static_assert(gemm_smem_bytes<kPleBN, kPleStages, EPI_PLE>() <= 232448, "PLE staging fits");
  return launch_gemm<kPleBN, kPleStages, EPI_PLE, kPleEpi>(a, tmY, tmW, tmEx, tmEx, a.B, kPleCols, kYD, 0, s);
}

cudaError_t launch_heads(const FwdArgs& a, const CUtensorMap& tmW1, cudaStream_t s) {
  return launch_kernel(heads_kernel, dim3((a.B + kBM - 1) / kBM, kNT), dim3(kThreads), kHeadSmem, s, a.pdl != 0, a, tmW1);
}

}  // namespace cvr
