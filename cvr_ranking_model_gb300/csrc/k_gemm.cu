// tcgen05 GEMMs of the CVR forward pass with fused epilogues: the tokeniser and the stacked layers' query FFNs.
//
//  gemm_kernel<EPI>  D[128 x BN] = A[128 x K] . W[BN x K]^T, both operands bf16 K-major in 128B-swizzled
//                    shared memory loaded by TMA through a STAGES-deep mbarrier ring; one elected thread
//                    issues tcgen05.mma into a TMEM accumulator; four epilogue warps drain TMEM with
//                    tcgen05.ld (one accumulator row per thread) and apply:
//    EPI_TOKENIZE    [Z[:, 0:1664] | Q] = bf16(I . [Wtok_item ; Wq_x Wtok_item]^T + [xu | qu + qb][request])
//                    (iQIYI 3.2.2 and 3.2.3 item 1): the tokens and, since the first layer's query FFN is
//                    linear in them, that layer's queries, with the query weights folded into the tokeniser
//                    (Wq_x Wtok precomputed). The per-request terms are computed once per request (iQIYI
//                    3.4.5): the user half xu = U . [Wtok_user ; Wq_x Wtok_user]^T + biases is the same GEMM
//                    over the pooled user rows, run as the first M-tiles of the launch (fp32 out); the item
//                    tiles' addends wait (bounded) for the xu tile of their requests and N-range, and the
//                    mean-pool term qb comes from the column-sum kernel
//    EPI_QUERY       Q = bf16(flat(X) . Wq_x^T + qb[request]) for stacked layers (iQIYI 3.2.3, item 1)
//
// The per-request addends of a tile are fetched one tile ahead by a warp of their own into shared memory (the
// request of each of the tile's rows, and the addend rows of up to kSlots consecutive requests), so the epilogue
// warps find them there instead of paying the request-id, flag and addend loads in series on every tile.
//
//  tokenize_lu_kernel  the tokeniser for batches of at most 32 requests ("lu": local user half): each CTA owns one
//                    column tile, keeps its weight slice in shared memory and computes that tile's user half for
//                    every request itself, so no CTA waits on another (used instead of gemm_kernel<EPI_TOKENIZE>)
#include "cvr_internal.cuh"

namespace cvr {

namespace {

enum { EPI_TOKENIZE = 0, EPI_QUERY = 1 };
constexpr int kBM = 128, kBK = 64;
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kSlots = 8;              // requests per tile whose addends are staged (others: loaded by the row)

// named barrier of the NEPI epilogue warps (the producer and MMA warps never take part); each warp arrives
// converged, since single lanes of it may have taken a branch of their own just before
template <int NEPI>
__device__ __forceinline__ void epi_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(NEPI * 32) : "memory");
}

template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() {
  return BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
}
// one addend buffer: the request of each row [128] int32, then kSlots addend rows [BN] fp32
template <int BN>
__host__ __device__ constexpr int add_buf_bytes() {
  return kBM * 4 + kSlots * BN * 4;
}
template <int BN, int STAGES, int EPI>
__host__ __device__ constexpr int gemm_smem_bytes() {
  return 1024 + STAGES * (kATile + BN * kBK * 2) + 256 +
         (EPI == EPI_TOKENIZE ? 1024 + 2 * kBM * BN * 2 : 0) +  // + output staging (aligned): two swizzled tiles
         2 * add_buf_bytes<BN>();                               // + two addend buffers
}

// v[0..32) += the addends of columns [nb, nb + 32) of a row of request `req`, read through L2: the tokeniser's
// xu + bias (+ the mean-pool term qb for the first layer's query columns), or the query GEMM's qb of the layer
template <int EPI>
__device__ __forceinline__ void add_row_addends(const FwdArgs& a, int req, int nb, int layer, float* v) {
  float t[32];
  if (EPI == EPI_TOKENIZE) {
    ldcg32(a.xu + (int64_t)req * kTokN + nb, t);  // (written in this launch)
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] += t[x];
    ldg32(a.tok_b + nb, t);
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] += t[x];
    if (nb >= kXD && !a.q_add) {
      ldg32(a.qb + (int64_t)req * (kG * kD) + (nb - kXD), t);
#pragma unroll
      for (int x = 0; x < 32; ++x) v[x] += t[x];
    }
  } else {
    ldg32(a.qb + ((int64_t)layer * a.R + req) * (kG * kD) + nb, t);
#pragma unroll
    for (int x = 0; x < 32; ++x) v[x] += t[x];
  }
}

// Persistent GEMM: CTAs loop over 128 x BN output tiles (n fastest, so co-running CTAs share A rows in L2).
// Warp 0 streams A/B k-blocks through a STAGES-deep ring; warp 1 issues the MMAs into one of two TMEM
// accumulators; NEPI epilogue warps drain the other one, so a tile's epilogue overlaps the next tile's
// MMAs. With 8 epilogue warps the two warpgroups split the 32-column chunks of a tile. The last warp stages
// the next row-tile's per-request addends in one of two shared-memory buffers.
template <int BN, int STAGES, int EPI, int NEPI>
__global__ void __launch_bounds__(96 + NEPI * 32, 1)
    gemm_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmZo,
                const __grid_constant__ CUtensorMap tmQo, const __grid_constant__ CUtensorMap tmU,
                const __grid_constant__ CUtensorMap tmWu, int M, int N, int K, int layer, int mu) {
  extern __shared__ uint8_t smem_raw[];
  CVR_TL_BEGIN(EPI == EPI_TOKENIZE ? TL_TOKENIZER : TL_QUERY);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int B_TILE = BN * kBK * 2;
  constexpr uint32_t TC = tmem_cols<BN>();
  constexpr int NCHUNK = (BN + 31) / 32;
  constexpr int NGRP = NEPI / 4;
  static_assert(BN <= 128, "one float4 of a tile row per lane of the addend warp");
  // TMEM accumulators: the tokeniser holds four (512 columns), so that the MMAs of a CTA's item tiles run on while
  // the epilogue waits for the user tile its first item tile needs; the query GEMM two
  constexpr int NACC = EPI == EPI_TOKENIZE ? 4 : 2;
  static_assert(NACC * TC <= 512, "accumulators fit tensor memory");
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * kATile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_TILE);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* add_full = acc_empty + NACC;  // addend buffer b staged
  uint64_t* add_empty = add_full + 2;   // addend buffer b read by every epilogue warp
  uint32_t* tslot = reinterpret_cast<uint32_t*>(add_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  // output staging for TMA stores (1024-byte aligned): tokeniser, two tiles [128][BN] bf16 as boxes of [128 rows]
  // [64 columns] with the 128-byte swizzle
  uint8_t* sOut = reinterpret_cast<uint8_t*>(((reinterpret_cast<uintptr_t>(full) + 256) + 1023) & ~uintptr_t(1023));
  uint8_t* sAdd = EPI == EPI_TOKENIZE ? sOut + 2 * kBM * BN * 2 : reinterpret_cast<uint8_t*>(full) + 256;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = N / BN;
  // tiles: mu user row-tiles (tokeniser only: xu = U . Wu^T), then the M rows; n fastest
  const int n_tiles = (mu + (M + kBM - 1) / kBM) * tiles_n;
  const int nk = K / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], NEPI);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&add_full[i], 1);
      mbar_init(&add_empty[i], NEPI);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tslot, NACC * TC);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();
  // The query GEMM's operand is the previous kernel's output: every warp waits for it. The tokeniser's copies need
  // no wait (the weights, and the gather kernel's rows, which are complete before this grid can launch: the
  // sequence encoder opens its edge only after its own wait for the gather kernel); its addend and epilogue warps,
  // which read the column sums' qb, wait for the previous grid while the first MMAs run.
  // (the query GEMM's producer issues its first stages' weights before it waits, below)
  if (EPI == EPI_TOKENIZE ? warp >= 2 : warp != 0) pdl_wait();
  if (threadIdx.x == (EPI == EPI_TOKENIZE ? 64 : 32)) CVR_TL_WAITED();

  if (warp == 0) {
    if (lane == 0) {
      int kc = 0, pre = 0;  // pre: k-blocks of the first tile whose weights are already in flight
      if (EPI == EPI_QUERY) {
        // the weights are constant: the first stages' copies start before the wait for the previous kernel
        if ((int)blockIdx.x < n_tiles) {
          pre = STAGES < nk ? STAGES : nk;
          for (int kb = 0; kb < pre; ++kb) {
            mbar_expect_tx(&full[kb], kATile + B_TILE);
            tma_load_2d(sB + kb * B_TILE, &tmB, &full[kb], kb * kBK, ((int)blockIdx.x % tiles_n) * BN);
          }
        }
        pdl_wait();
      }
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int mt = tile / tiles_n, n0 = (tile % tiles_n) * BN;
        const bool user = mt < mu;
        const int m0 = (user ? mt : mt - mu) * kBM;
        for (int kb = 0; kb < nk; ++kb, ++kc) {
          const int s = kc % STAGES;
          if (kc >= STAGES && !mbar_wait(&empty[s], ((kc / STAGES) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          if (kc >= pre) mbar_expect_tx(&full[s], kATile + B_TILE);
          tma_load_2d(sA + s * kATile, user ? &tmU : &tmA, &full[s], kb * kBK, m0);
          if (kc >= pre) tma_load_2d(sB + s * B_TILE, user ? &tmWu : &tmB, &full[s], kb * kBK, n0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, BN);
      int kc = 0, i = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++i) {
        const int buf = i % NACC;
        if (i >= NACC && !mbar_wait(&acc_empty[buf], ((i / NACC) & 1) ^ 1, abort_flag, a.err)) break;
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
  } else if (warp == 2 + NEPI) {
    // ---- addends of the row-tiles, ahead of the epilogue: the request of every row, then for the tile's first
    // kSlots requests (rows are sorted by request) the addend row xu (+ qb for the first layer's query columns), or
    // qb of the layer; the tokeniser waits (bounded) for the user tile that writes xu. Each step is one round trip
    // to memory: the next tile's request ids are loaded while this tile's addends are, and a flag seen set is
    // remembered.
    auto next_item = [&](int t) {
      while (t < n_tiles && EPI == EPI_TOKENIZE && t / tiles_n < mu) t += gridDim.x;
      return t;
    };
    int rq[kBM / 32];  // request ids of this lane's rows of the next tile
    auto load_req = [&](int t) {
      const int m0 = (t / tiles_n - mu) * kBM;
#pragma unroll
      for (int k = 0; k < kBM / 32; ++k) {
        const int row = m0 + lane + 32 * k;
        rq[k] = row < M ? a.req_ids[row] : 0;
      }
    };
    int tile = next_item(blockIdx.x), j = 0, flag_seen = -1;
    if (tile < n_tiles) load_req(tile);
    while (tile < n_tiles) {
      const int mt = tile / tiles_n, nt = tile % tiles_n, n0 = nt * BN;
      const int b = j & 1;
      if (j >= 2 && !mbar_wait_warp(&add_empty[b], ((j >> 1) & 1) ^ 1, abort_flag, a.err)) break;
      const int m0 = (mt - mu) * kBM;
      int* sreq = reinterpret_cast<int*>(sAdd + b * add_buf_bytes<BN>());
      float* sadd = reinterpret_cast<float*>(sreq + kBM);
#pragma unroll
      for (int k = 0; k < kBM / 32; ++k) sreq[lane + 32 * k] = min(max(rq[k], 0), a.R - 1);
      __syncwarp();
      const int nxt = next_item(tile + gridDim.x);
      if (nxt < n_tiles) load_req(nxt);  // (in flight while this tile's addends load)
      const int r_first = sreq[0];
      const int n_slots = max(0, min(kSlots, sreq[min(M - m0, kBM) - 1] - r_first + 1));
      bool ok = true;
      if (EPI == EPI_TOKENIZE) {
        for (int sl = 0; sl < n_slots && ok; ++sl) {
          const int fi = ((r_first + sl) / kBM) * tiles_n + nt;  // one flag per 128 requests and column tile
          if (fi == flag_seen) continue;
          const unsigned* flag = a.xu_ready + fi;
          if (ld_acquire_u32(flag) == 0u) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_u32(flag) == 0u) {
              if (*abort_flag || global_timer_ns() - t0 > 1000000000ull) {
                atomicOr(a.err, kErrTimeout);
                ok = false;
                break;
              }
              __nanosleep(32);
            }
          }
          flag_seen = fi;
        }
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      for (int s0 = 0; s0 < n_slots; s0 += 4) {  // four addend rows in flight at a time
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int sl = s0 + k, r = r_first + sl, x = lane * 4;
        if (sl >= n_slots || x >= BN) continue;
        if (EPI == EPI_TOKENIZE) {
          v[k] = __ldcg(reinterpret_cast<const float4*>(a.xu + (int64_t)r * kTokN + n0 + x));  // (written in this launch)
          const float4 bv = __ldg(reinterpret_cast<const float4*>(a.tok_b + n0 + x));
          v[k] = make_float4(v[k].x + bv.x, v[k].y + bv.y, v[k].z + bv.z, v[k].w + bv.w);
          if (n0 >= kXD && !a.q_add) {  // first-layer query columns: + the mean-pool term of the request
            const float4 qv = __ldg(reinterpret_cast<const float4*>(a.qb + (int64_t)r * (kG * kD) + (n0 - kXD) + x));
            v[k] = make_float4(v[k].x + qv.x, v[k].y + qv.y, v[k].z + qv.z, v[k].w + qv.w);
          }
        } else {
          v[k] = __ldg(reinterpret_cast<const float4*>(a.qb + ((int64_t)layer * a.R + r) * (kG * kD) + n0 + x));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (s0 + k < n_slots && lane * 4 < BN) *reinterpret_cast<float4*>(sadd + (s0 + k) * BN + lane * 4) = v[k];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&add_full[b]);
      tile = nxt;
      ++j;
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;     // chunk group
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int i = 0, j = 0;  // tiles, row-tiles (addend buffers)
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
      const int mt = tile / tiles_n, nt = tile % tiles_n, n0 = nt * BN;
      const int buf = i % NACC;
      constexpr int NMY = (NCHUNK + NGRP - 1) / NGRP;
      if (EPI == EPI_TOKENIZE && mt < mu) {
        // user row-tile: xu[r][n0 + ..] = acc, fp32 (the bias is added with it by the item tiles); then the tile is
        // published to the item tiles
        const int r = mt * kBM + q * 32 + lane;
        if (!mbar_wait(&acc_full[buf], (i / NACC) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        uint32_t acc[NMY][32];
#pragma unroll
        for (int m = 0; m < NMY; ++m)
          if (grp + m * NGRP < NCHUNK) tmem_ld32_nowait(tbase + lane_off + buf * TC + (grp + m * NGRP) * 32, acc[m]);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < NMY; ++m) {
          const int c = grp + m * NGRP;
          if (c >= NCHUNK || r >= a.R) continue;
          const float* v = reinterpret_cast<const float*>(acc[m]);
          float4* dst = reinterpret_cast<float4*>(a.xu + (int64_t)r * kTokN + n0 + c * 32);
#pragma unroll
          for (int x = 0; x < 8; ++x) dst[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        epi_bar<NEPI>();
        // the barrier orders every warp's xu stores before this release (cumulativity)
        if (threadIdx.x == 64) red_release_add(a.xu_ready + mt * tiles_n + nt, 1u);
        continue;
      }
      const int m0 = (mt - mu) * kBM;
      const int rl = q * 32 + lane, row = m0 + rl;
      const bool live = row < M;
      const int b = j & 1;
      const bool staged_ok = mbar_wait_warp(&add_full[b], (j >> 1) & 1, abort_flag, a.err);
      const int* sreq = reinterpret_cast<const int*>(sAdd + b * add_buf_bytes<BN>());
      const float* sadd = reinterpret_cast<const float*>(sreq + kBM);
      const int req = live ? sreq[rl] : 0;
      const int n_slots = max(0, min(kSlots, sreq[min(M - m0, kBM) - 1] - sreq[0] + 1));
      const int slot = req - sreq[0];
      const bool staged = slot >= 0 && slot < n_slots;
      if (EPI == EPI_TOKENIZE && live && !staged && staged_ok) {
        // a request past the staged ones: its user tile is waited for here (bounded)
        const unsigned* flag = a.xu_ready + (req / kBM) * tiles_n + nt;
        if (ld_acquire_u32(flag) == 0u) {
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_u32(flag) == 0u) {
            if (*abort_flag || global_timer_ns() - t0 > 1000000000ull) {
              atomicOr(a.err, kErrTimeout);
              break;
            }
            __nanosleep(32);
          }
        }
      }
      if (!staged_ok || !mbar_wait_warp(&acc_full[buf], (i / NACC) & 1, abort_flag, a.err)) break;
      tc_fence_after();
      uint8_t* sb = sOut + (i & 1) * (kBM * BN * 2);
      if (EPI == EPI_TOKENIZE) {
        // the TMA store issued from this staging buffer earlier must have finished reading it
        if (threadIdx.x == 64) bulk_wait_read<1>();
        epi_bar<NEPI>();
      }
#pragma unroll
      for (int m = 0; m < NMY; ++m) {
        const int c = grp + m * NGRP;
        if (c >= NCHUNK) continue;
        float v[32];
        tmem_ld32(tbase + lane_off + buf * TC + c * 32, v);
        const int nb = n0 + c * 32;
        if (!live) continue;
        // v += the row's addends: staged in shared memory, else (a request past the staged ones) read through L2
        if (staged) {
          const float4* ap = reinterpret_cast<const float4*>(sadd + slot * BN + c * 32);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float4 t = ap[x];
            v[4 * x] += t.x;
            v[4 * x + 1] += t.y;
            v[4 * x + 2] += t.z;
            v[4 * x + 3] += t.w;
          }
        } else {
          add_row_addends<EPI>(a, req, nb, layer, v);
        }
        if (EPI == EPI_TOKENIZE) {
          // columns [32c, 32c + 32) of row rl into the staging tile: box c/2, 16-byte chunks 4 (c%2) + j, swizzled
          uint8_t* rowp = sb + (c >> 1) * (kBM * 128) + rl * 128;
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            uint4 p;
            p.x = pack_bf16(v[8 * j4 + 0], v[8 * j4 + 1]);
            p.y = pack_bf16(v[8 * j4 + 2], v[8 * j4 + 3]);
            p.z = pack_bf16(v[8 * j4 + 4], v[8 * j4 + 5]);
            p.w = pack_bf16(v[8 * j4 + 6], v[8 * j4 + 7]);
            *reinterpret_cast<uint4*>(rowp + ((((c & 1) * 4 + j4) ^ (rl & 7)) << 4)) = p;
          }
        } else if (EPI == EPI_QUERY) {
          __nv_bfloat16* out = a.Q + (int64_t)row * (kG * kD) + nb;
          uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            if (c * 32 + j4 * 8 >= BN) break;
            uint4 p;
            p.x = pack_bf16(v[8 * j4 + 0], v[8 * j4 + 1]);
            p.y = pack_bf16(v[8 * j4 + 2], v[8 * j4 + 3]);
            p.z = pack_bf16(v[8 * j4 + 4], v[8 * j4 + 5]);
            p.w = pack_bf16(v[8 * j4 + 6], v[8 * j4 + 7]);
            dst[j4] = p;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&add_empty[b]);  // (this warp is done with the addend buffer)
      ++j;
      if (EPI == EPI_TOKENIZE) {
        // the whole tile is staged: one thread stores it in boxes of 64 columns, tokens into Z and the first
        // layer's queries into Q
        fence_proxy_async_smem();
        epi_bar<NEPI>();
        if (threadIdx.x == 64) {
          const bool qcols = n0 >= kXD;
#pragma unroll
          for (int bx = 0; bx < BN / 64; ++bx)
            tma_store_2d(qcols ? &tmQo : &tmZo, sb + bx * (kBM * 128), (qcols ? n0 - kXD : n0) + bx * 64, m0);
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    // (the staging buffers have been read before the CTA exits; the stores complete with the grid, which the next
    // kernel waits for)
    if (EPI == EPI_TOKENIZE && threadIdx.x == 64) bulk_wait_read<0>();
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, NACC * TC);
  }
}

// ------------------------------------------------------------------------------------------
// The tokeniser for batches of at most kLuMaxR requests. The grid is a multiple of the 16 column tiles, so each
// CTA owns one column tile n0 for all of its row-tiles:
//  - its weight slice Wtok_item[n0, n0 + 128) (K = 256, 64 KB) is loaded once and stays in shared memory; only the
//    A k-blocks (16 KB) stream through the stage ring (the main loop is bound by shared-memory bandwidth, not by
//    the tensor pipe, so every byte that does not pass through shared memory counts);
//  - it computes the user half of its column tile for every request itself, transposed:
//    xu^T = Wu[n0 ..] . U^T (M = 128 output columns, N = 32 requests, K = 256) into 32 TMEM columns, adds the bias
//    (and the first layer's mean-pool term qb when the attention does not add it) and keeps it in shared memory,
//    so no item tile waits on another CTA (iQIYI 3.4.5: the user side once per request, here once per CTA). Its
//    MMAs follow the first row-tile's, whose operands are loaded first.
// Warp 0: TMA; warp 1: MMA issue; warps 2..2+NEPI-1: epilogue; the last warp stages each row-tile's request ids.
// Output: one 128B-swizzled staging tile stored by TMA (it holds the user rows until the user half is done).
constexpr int kLuMaxR = kTokOwnXuMaxR;
constexpr int kLuStages = 7;
constexpr int kLuEpi = 8;
constexpr int kLuUBytes = kLuMaxR * kBK * 2;  // one k-block of the user rows: [32][64] bf16

struct LuSmem {  // byte offsets from the 1024-aligned base
  static constexpr int kA = 0;                                  // kLuStages x [128][64] bf16
  static constexpr int kB = kA + kLuStages * kATile;            // the CTA's weight slice: 4 x [128][64] bf16
  static constexpr int kOut = kB + (kID / kBK) * kATile;        // staging [128][128] bf16 (two 64-column boxes);
                                                                 // first the user rows: 4 x [32][64] bf16
  static constexpr int kXu = kOut + kBM * 128 * 2;              // xu + bias (+ qb) [kLuMaxR][128] fp32
  static constexpr int kReq = kXu + kLuMaxR * 128 * 4;          // request ids of two row-tiles [2][128] int32
  static constexpr int kBar = kReq + 2 * kBM * 4;
  static constexpr int kNBar = 2 * kLuStages + 2 * 4 + 1 + 2 + 2;
  static constexpr int kBytes = 1024 + kBar + kNBar * 8 + 16;
};
static_assert(LuSmem::kBytes <= 232448, "shared memory budget of one CTA");
static_assert((kUD / kBK) * kLuUBytes <= kBM * 128 * 2, "the user rows fit the staging tile");

template <int NEPI>
__global__ void __launch_bounds__(96 + NEPI * 32, 1)
    tokenize_lu_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmZo,
                       const __grid_constant__ CUtensorMap tmQo, const __grid_constant__ CUtensorMap tmU32,
                       const __grid_constant__ CUtensorMap tmWu) {
  extern __shared__ uint8_t smem_raw[];
  CVR_TL_BEGIN(TL_TOKENIZER);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int BN = 128, NCHUNK = BN / 32, NGRP = NEPI / 4, NMY = NCHUNK / NGRP, NACC = 4, nk = kID / kBK;
  static_assert(NEPI == 8 && 16 * NGRP == kLuMaxR, "each epilogue warpgroup drains 16 requests of the user half");
  static_assert(kUD == kID, "the user half and the item tiles share the k-block count");
  uint8_t* sA = smem + LuSmem::kA;
  uint8_t* sB = smem + LuSmem::kB;
  uint8_t* sOut = smem + LuSmem::kOut;
  uint8_t* sU = sOut;  // (until the user half's MMAs are done)
  float* sXu = reinterpret_cast<float*>(smem + LuSmem::kXu);
  int* sReq = reinterpret_cast<int*>(smem + LuSmem::kReq);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LuSmem::kBar);
  uint64_t* empty = full + kLuStages;
  uint64_t* acc_full = empty + kLuStages;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* bres_full = acc_empty + NACC;  // the weight slice landed
  uint64_t* req_full = bres_full + 1;      // request ids of row-tile buffer b staged
  uint64_t* req_empty = req_full + 2;      // ... and read by every epilogue warp
  uint32_t* tslot = reinterpret_cast<uint32_t*>(req_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.B;
  constexpr int tiles_n = kTokN / BN;
  const int n_tiles = (M + kBM - 1) / kBM * tiles_n;
  const int n0 = (int)(blockIdx.x % tiles_n) * BN;  // (gridDim.x % tiles_n == 0)
  // Jobs in ring and MMA order: the first row-tile (if any), the user half, the other row-tiles. Accumulator use u
  // (buffer u % NACC): the user half u = 0, the k-th row-tile u = k + 1.
  const int n_items = (int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int xu_job = n_items > 0 ? 1 : 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kLuStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], NEPI);
    }
    mbar_init(bres_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&req_full[i], 1);
      mbar_init(&req_empty[i], NEPI);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmU32);
    tma_prefetch_desc(&tmWu);
  }
  if (warp == 1) tmem_alloc(tslot, NACC * BN);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // The copies need no wait for the previous kernel: the weights are constant, and the item and user rows
      // come from the gather kernel, which has completed before this grid can launch (the side stream starts
      // after it; on one stream the sequence encoder opens its edge only after its own wait for it). Only the
      // epilogue, which adds the column sums' qb, waits for the previous grid; the MMAs run meanwhile.
      mbar_expect_tx(bres_full, nk * kATile);
      for (int kb = 0; kb < nk; ++kb) tma_load_2d(sB + kb * kATile, &tmB, bres_full, kb * kBK, n0);
      int kc = 0;
      bool ok = true;
      for (int job = 0; job < n_items + 1 && ok; ++job) {
        const bool xu = job == xu_job;
        const int m0 = ((int)blockIdx.x + (job - (job > xu_job)) * (int)gridDim.x) / tiles_n * kBM;
        for (int kb = 0; kb < nk; ++kb, ++kc) {
          const int s = kc % kLuStages;
          if (kc >= kLuStages && !mbar_wait(&empty[s], ((kc / kLuStages) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          if (xu) {  // A = Wu rows [n0, n0 + 128), B = U rows [0, 32)
            mbar_expect_tx(&full[s], kATile + kLuUBytes);
            tma_load_2d(sA + s * kATile, &tmWu, &full[s], kb * kBK, n0);
            tma_load_2d(sU + kb * kLuUBytes, &tmU32, &full[s], kb * kBK, 0);
          } else {
            mbar_expect_tx(&full[s], kATile);
            tma_load_2d(sA + s * kATile, &tmA, &full[s], kb * kBK, m0);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_xu = idesc_bf16(kBM, kLuMaxR), id_it = idesc_bf16(kBM, BN);
      bool ok = mbar_wait(bres_full, 0, abort_flag, a.err);
      int kc = 0;
      for (int job = 0; job < n_items + 1 && ok; ++job) {
        const bool xu = job == xu_job;
        const int u = xu ? 0 : job + (job < xu_job), buf = u % NACC;
        if (u >= NACC && !mbar_wait(&acc_empty[buf], ((u / NACC) & 1) ^ 1, abort_flag, a.err)) break;
        const uint32_t dacc = tbase + buf * BN;
        for (int kb = 0; kb < nk; ++kb, ++kc) {
          const int s = kc % kLuStages;
          if (!mbar_wait(&full[s], (kc / kLuStages) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aa = smem_u32(sA + s * kATile);
          const uint32_t bb = xu ? smem_u32(sU + kb * kLuUBytes) : smem_u32(sB + kb * kATile);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma(dacc, sdesc_sw128(aa + k * 32), sdesc_sw128(bb + k * 32), xu ? id_xu : id_it, (kb | k) != 0);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&acc_full[buf]);
      }
    }
  } else if (warp == 2 + NEPI) {
    // ---- request ids of each row-tile (clamped into [0, R); the sparse kernel reports bad ones), one tile ahead
    // (the gather kernel's copy: complete before this grid launches, as the rows above)
    int rq[kBM / 32];
    auto load_req = [&](int t) {
      const int m0 = (t / tiles_n) * kBM;
#pragma unroll
      for (int k = 0; k < kBM / 32; ++k) {
        const int row = m0 + lane + 32 * k;
        rq[k] = row < M ? a.req_ids[row] : 0;
      }
    };
    int tile = blockIdx.x, j = 0;
    if (tile < n_tiles) load_req(tile);
    for (; tile < n_tiles; tile += gridDim.x, ++j) {
      const int b = j & 1;
      if (j >= 2 && !mbar_wait_warp(&req_empty[b], ((j >> 1) & 1) ^ 1, abort_flag, a.err)) break;
#pragma unroll
      for (int k = 0; k < kBM / 32; ++k) sReq[b * kBM + lane + 32 * k] = min(max(rq[k], 0), a.R - 1);
      __syncwarp();
      if (tile + (int)gridDim.x < n_tiles) load_req(tile + gridDim.x);  // (in flight until the next tile)
      if (lane == 0) mbar_arrive(&req_full[b]);
    }
  } else {
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;  // chunk group
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    // user half: TMEM lane n = output column n0 + n, column r = request r; this warpgroup drains requests
    // [16 grp, 16 grp + 16). Its addends are loaded before the wait. Every warp arrives and meets at the barrier,
    // whatever its wait returned.
    const int n = q * 32 + lane, nb = n0 + n;
    const float bias = __ldg(a.tok_b + nb);
    pdl_wait();  // (qb, when it is added here, comes from the column-sum kernel)
    if (threadIdx.x == 64) CVR_TL_WAITED();
    const bool addq = nb >= kXD && !a.q_add;
    float qv[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const int r = grp * 16 + x;
      qv[x] = addq && r < a.R ? __ldg(a.qb + (int64_t)r * (kG * kD) + (nb - kXD)) : 0.f;
    }
    bool ok = mbar_wait_warp(&acc_full[0], 0, abort_flag, a.err);
    if (ok) {
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16_nowait(tbase + lane_off + grp * 16, v);
      tmem_ld_wait();
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int r = grp * 16 + x;
        float t = __uint_as_float(v[x]) + bias;
        if (addq) t += qv[x];
        if (r < a.R) sXu[r * BN + n] = t;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&acc_empty[0]);
    epi_bar<NEPI>();
    int u = 1, j = 0;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++u, ++j) {
      const int m0 = (tile / tiles_n) * kBM;
      const int rl = q * 32 + lane, row = m0 + rl;
      const bool live = row < M;
      const int buf = u % NACC, b = j & 1;
      if (!mbar_wait_warp(&req_full[b], (j >> 1) & 1, abort_flag, a.err) ||
          !mbar_wait_warp(&acc_full[buf], (u / NACC) & 1, abort_flag, a.err))
        break;
      tc_fence_after();
      const float* xr = sXu + sReq[b * kBM + rl] * BN;
      __syncwarp();
      if (lane == 0) mbar_arrive(&req_empty[b]);
      // the previous tile's TMA store has finished reading the staging tile (before the first tile, the user half's
      // MMAs, which read the user rows kept there, have completed: its accumulator was drained above)
      if (threadIdx.x == 64) bulk_wait_read<0>();
      epi_bar<NEPI>();
#pragma unroll
      for (int m = 0; m < NMY; ++m) {
        const int c = grp + m * NGRP;
        float v[32];
        tmem_ld32(tbase + lane_off + buf * BN + c * 32, v);
        if (m == NMY - 1) {  // the accumulator is read: the MMAs may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (!live) continue;
        const float4* ap = reinterpret_cast<const float4*>(xr + c * 32);
        // columns [32c, 32c + 32) of row rl into the staging tile: box c/2, 16-byte chunks 4 (c%2) + j4, swizzled
        uint8_t* rowp = sOut + (c >> 1) * (kBM * 128) + rl * 128;
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 t0 = ap[2 * j4], t1 = ap[2 * j4 + 1];
          uint4 p;
          p.x = pack_bf16(v[8 * j4 + 0] + t0.x, v[8 * j4 + 1] + t0.y);
          p.y = pack_bf16(v[8 * j4 + 2] + t0.z, v[8 * j4 + 3] + t0.w);
          p.z = pack_bf16(v[8 * j4 + 4] + t1.x, v[8 * j4 + 5] + t1.y);
          p.w = pack_bf16(v[8 * j4 + 6] + t1.z, v[8 * j4 + 7] + t1.w);
          *reinterpret_cast<uint4*>(rowp + ((((c & 1) * 4 + j4) ^ (rl & 7)) << 4)) = p;
        }
      }
      fence_proxy_async_smem();
      epi_bar<NEPI>();
      if (threadIdx.x == 64) {
        const bool qcols = n0 >= kXD;
#pragma unroll
        for (int bx = 0; bx < BN / 64; ++bx)
          tma_store_2d(qcols ? &tmQo : &tmZo, sOut + bx * (kBM * 128), (qcols ? n0 - kXD : n0) + bx * 64, m0);
        bulk_commit();
      }
    }
    // (the staging tile has been read before the CTA exits; the stores complete with the grid)
    if (threadIdx.x == 64) bulk_wait_read<0>();
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, NACC * BN);
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
                        const CUtensorMap& tmQo, const CUtensorMap& tmU, const CUtensorMap& tmWu, int M, int N, int K,
                        int layer, int mu, cudaStream_t s, int max_grid = 0, bool pdl = true) {
  const int tiles = (mu + (M + kBM - 1) / kBM) * (N / BN);
  const int cap = max_grid > 0 && max_grid < a.num_sms ? max_grid : a.num_sms;
  const int grid = tiles < cap ? tiles : cap;
  return launch_kernel(gemm_kernel<BN, STAGES, EPI, NEPI>, dim3(grid), dim3(96 + NEPI * 32), gemm_smem_bytes<BN, STAGES, EPI>(),
                       s, pdl && a.pdl != 0, a, tmA, tmB, tmZo, tmQo, tmU, tmWu, M, N, K, layer, mu);
}

constexpr int kTokBN = 128, kTokStages = 4, kTokEpi = 8;
constexpr int kQryStages = 6, kQryEpi = 8;
static_assert((kG * kD) % kQryBNNarrow == 0 && (kG * kD) % kQryBNWide == 0, "both query tile widths divide Q's columns");

}  // namespace

cudaError_t prepare_gemm_kernels() {
  cudaError_t e = prepare_gemm<kTokBN, kTokStages, EPI_TOKENIZE, kTokEpi>();
  if (e == cudaSuccess) e = prepare_gemm<kQryBNNarrow, kQryStages, EPI_QUERY, kQryEpi>();
  if (e == cudaSuccess) e = prepare_gemm<kQryBNWide, kQryStages, EPI_QUERY, kQryEpi>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tokenize_lu_kernel<kLuEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize, LuSmem::kBytes);
  return e;
}

cudaError_t launch_tokenizer(const FwdArgs& a, const CUtensorMap& tmI, const CUtensorMap& tmW, const CUtensorMap& tmZo,
                             const CUtensorMap& tmQo, const CUtensorMap& tmU, const CUtensorMap& tmU32,
                             const CUtensorMap& tmWu, int max_grid, bool pdl, cudaStream_t s) {
  static_assert(kXD % kTokBN == 0 && kTokN % kTokBN == 0, "token and query columns fall in separate tiles");
  static_assert(kTokBN % 64 == 0 && gemm_smem_bytes<kTokBN, kTokStages, EPI_TOKENIZE>() <= 232448, "staging fits");
  constexpr int tiles_n = kTokN / 128;
  const int cap = max_grid > 0 && max_grid < a.num_sms ? max_grid : a.num_sms;
  if (a.R <= kLuMaxR && cap >= tiles_n) {  // each CTA one column tile, its own user half
    const int tiles = (a.B + kBM - 1) / kBM * tiles_n;
    int grid = tiles < cap ? tiles : cap;
    grid -= grid % tiles_n;
    return launch_kernel(tokenize_lu_kernel<kLuEpi>, dim3(grid), dim3(96 + kLuEpi * 32), LuSmem::kBytes, s,
                         pdl && a.pdl != 0, a, tmI, tmW, tmZo, tmQo, tmU32, tmWu);
  }
  return launch_gemm<kTokBN, kTokStages, EPI_TOKENIZE, kTokEpi>(a, tmI, tmW, tmZo, tmQo, tmU, tmWu, a.B, kTokN, kID, 0,
                                                                (a.R + kBM - 1) / kBM, s, max_grid, pdl);
}

cudaError_t launch_query(const FwdArgs& a, int layer, const CUtensorMap& tmX, const CUtensorMap& tmW,
                         const CUtensorMap& tmWw, cudaStream_t s) {
  // The main loop is bound by shared memory: a k-block moves A (16 KB) and B (BN rows x 128 B) through it. Wide
  // tiles move fewer bytes per column but make fewer, longer tiles: take the width whose rounds of tiles over the
  // persistent grid cost fewer bytes (wide from 512 candidates per 152 SMs upwards).
  auto cost = [&](int bn) {
    const int64_t tiles = (int64_t)((a.B + kBM - 1) / kBM) * (kG * kD / bn);
    const int64_t grid = tiles < a.num_sms ? tiles : a.num_sms;
    return (tiles + grid - 1) / grid * (int64_t)(kATile + bn * kBK * 2);
  };
  if (cost(kQryBNWide) < cost(kQryBNNarrow))
    return launch_gemm<kQryBNWide, kQryStages, EPI_QUERY, kQryEpi>(a, tmX, tmWw, tmX, tmX, tmX, tmX, a.B, kG * kD, kXD,
                                                                    layer, 0, s);
  return launch_gemm<kQryBNNarrow, kQryStages, EPI_QUERY, kQryEpi>(a, tmX, tmW, tmX, tmX, tmX, tmX, a.B, kG * kD, kXD,
                                                                    layer, 0, s);
}

}  // namespace cvr
