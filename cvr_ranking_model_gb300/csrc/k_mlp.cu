// Fused SwiGLU 128 -> 256 -> 128 on tcgen05, used twice in the CVR forward pass:
//
//  SEQ  the per-group sequence encoder (iQIYI ad-CVR article 3.2.2: each behaviour sequence is mapped
//       position-wise into the token space by its own SwiGLU): rows = sequence events of one group,
//       output H = W2 (silu(W1 x + b1) * (W3 x + b3)) + b2.
//  TM   the Query Boosting Token Mixer (iQIYI 3.2.3): the A operand is Mix(Z) -- 16 tokens x 16 heads of
//       8 transposed -- which the TMA unit writes into shared memory straight from Z through a 5-D tensor
//       map (token t, head j of candidate b becomes K-slot t of mixed row (b, j)); the epilogue applies the
//       inverse map (Revert), the residual and the RMSNorm and writes Y in the original token order.
//
// Persistent and warp-specialised: one CTA per SM loops over 128-row tiles. All SwiGLU weights (W1/W3 128 KB,
// W2 64 KB) stay resident in shared memory -- only the 32 KB activation tile crosses L2 per tile (reloaded
// only when a sequence tile changes group). The hidden width is processed in 4 chunks of 64 units: the up
// projection of chunk c is one N=128 MMA chain (64 W1 rows + 64 W3 rows, K=128) into a TMEM up-buffer;
// eight epilogue warps turn it into silu(a)*g and store the bf16 hidden chunk back into TMEM, where it is
// the A operand of the down projection (4 MMAs, K=64, B = the matching 64 columns of W2) accumulating into
// the TMEM down-buffer. The MMA warp issues the up projection two chunks ahead of the down projection, so
// the tensor pipe works while the epilogue computes. TMEM: up 2 x 128, down 128, hidden 2 x 32 columns.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;   // warp 0: TMA, warp 1: MMA, warps 2..9: epilogue
constexpr int kChunks = 4;                      // hidden chunks of 64
constexpr int kATile = 128 * kD * 2;            // 32 KB
constexpr int kW13Bytes = 2 * kHid * kD * 2;    // 128 KB: chunk c = [W1 64 rows ; W3 64 rows] x 128, 2 K-blocks
constexpr int kW2Bytes = kD * kHid * 2;         // 64 KB: 4 K-blocks of [128][64]
constexpr int kOffA = 0;
constexpr int kOffW13 = kOffA + kATile;
constexpr int kOffW2 = kOffW13 + kW13Bytes;
constexpr int kOffBias = kOffW2 + kW2Bytes;     // fp32 b1/b3 [512] (chunk-interleaved) + b2 [128] of one group
constexpr int kBiasFloats = 2 * kHid + kD;
constexpr int kOffBar = kOffBias + kBiasFloats * 4;
constexpr int kNBar = 4 + 4 * 2 + 2;
// The dynamic shared-memory window is 1024-byte aligned (checked at run time; the kernel reports an error
// and does nothing otherwise), so no alignment slack is requested: the whole 227 KB budget is used.
constexpr int kSmemBytes = kOffBar + kNBar * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
constexpr uint32_t kColUp = 0, kColDown = 256, kColHid = 384;  // TMEM column bases

enum { MODE_SEQ = 0, MODE_TM = 1 };

struct TileInfo {
  int g;
  int64_t row0, rows_end;
};

template <int MODE>
__device__ __forceinline__ TileInfo tile_info(const FwdArgs& a, int tile) {
  TileInfo ti;
  if (MODE == MODE_SEQ) {
    int g = 0;
    while (g < kG - 1) {
      const int tg = (int)(((int64_t)a.R * a.L[g] + 127) / 128);
      if (tile < tg) break;
      tile -= tg;
      ++g;
    }
    ti.g = g;
    ti.row0 = a.goff[g] + (int64_t)tile * 128;
    ti.rows_end = a.goff[g] + (int64_t)a.R * a.L[g];
  } else {
    ti.g = 0;
    ti.row0 = (int64_t)tile * 128;
    ti.rows_end = (int64_t)a.B * kT;
  }
  return ti;
}

// Named barrier among the epilogue warps only (the producer and MMA warps never take part).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory"); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    swiglu_mlp_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2, int layer,
                      int n_tiles, const __nv_bfloat16* __restrict__ zin, __nv_bfloat16* __restrict__ yout) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrLayout);
    return;
  }
  uint8_t* sA = smem + kOffA;
  uint8_t* sW13 = smem + kOffW13;
  uint8_t* sW2 = smem + kOffW2;
  float* sb13 = reinterpret_cast<float*>(smem + kOffBias);
  float* sb2 = sb13 + 2 * kHid;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bar;              // activation tile landed
  uint64_t* a_empty = bar + 1;         // last up MMA of the tile has read it
  uint64_t* w_full = bar + 2;          // weights landed
  uint64_t* w_empty = bar + 3;         // weights may be replaced (sequence group change)
  uint64_t* up_full = bar + 4;         // [2] up accumulator ready
  uint64_t* up_empty = bar + 6;        // [2] epilogue has read it
  uint64_t* hm_full = bar + 8;         // [2] hidden chunk stored in TMEM
  uint64_t* hm_empty = bar + 10;       // [2] down MMAs have read it
  uint64_t* dn_full = bar + 12;        // down accumulator ready
  uint64_t* dn_empty = bar + 13;       // epilogue has read it
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    mbar_init(w_full, 1);
    mbar_init(w_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&up_full[i], 1);
      mbar_init(&up_empty[i], kEpiWarps);
      mbar_init(&hm_full[i], kEpiWarps);
      mbar_init(&hm_empty[i], 1);
    }
    mbar_init(dn_full, 1);
    mbar_init(dn_empty, kEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW13);
    tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_trigger();
  const int n_my = blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Weights are constant, so their loads may start before the previous kernel has finished; the
      // activation loads wait for it (pdl_wait) first.
      int w_group = -1, w_loads = 0;
      bool waited = false;
      for (int i = 0; i < n_my; ++i) {
        const TileInfo ti = tile_info<MODE>(a, blockIdx.x + i * gridDim.x);
        if (ti.g != w_group) {  // (TM: once)
          if (w_loads > 0 && !mbar_wait(w_empty, (w_loads - 1) & 1, abort_flag, a.err)) break;
          const int wsel = MODE == MODE_SEQ ? ti.g : layer;
          mbar_expect_tx(w_full, kW13Bytes + kW2Bytes);
          for (int c = 0; c < kChunks; ++c) {
            tma_load_2d(sW13 + c * 32768, &tmW13, w_full, 0, wsel * 2 * kHid + c * 128);
            tma_load_2d(sW13 + c * 32768 + 16384, &tmW13, w_full, 64, wsel * 2 * kHid + c * 128);
          }
          for (int kb = 0; kb < 4; ++kb) tma_load_2d(sW2 + kb * 16384, &tmW2, w_full, kb * 64, wsel * kD);
          w_group = ti.g;
          ++w_loads;
        }
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        if (i >= 1 && !mbar_wait(a_empty, (i - 1) & 1, abort_flag, a.err)) break;
        mbar_expect_tx(a_full, kATile);
        if (MODE == MODE_SEQ) {
          tma_load_2d(sA, &tmA, a_full, 0, (int)ti.row0);
          tma_load_2d(sA + kATile / 2, &tmA, a_full, 64, (int)ti.row0);
        } else {
          // Z[b][t][8j+e] -> smem [b][j/8][t][j%8][e]: core matrices of 8 mixed rows x 8 K-elements
          tma_load_5d(sA, &tmA, a_full, 0, 0, 0, 0, (int)(ti.row0 / kT));
        }
      }
      if (!waited) pdl_wait();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id128 = idesc_bf16(128, 128);
      const int total = n_my * kChunks;
      int w_group = -1, w_loads = 0;
      bool ok = true;
      auto issue_up = [&](int cc) -> bool {
        const int i = cc / kChunks, c = cc % kChunks, u = cc & 1;
        if (c == 0) {
          const int g = tile_info<MODE>(a, blockIdx.x + i * gridDim.x).g;
          if (g != w_group) {
            if (!mbar_wait(w_full, w_loads & 1, abort_flag, a.err)) return false;
            w_group = g;
            ++w_loads;
          }
          if (!mbar_wait(a_full, i & 1, abort_flag, a.err)) return false;
        }
        if (cc >= 2 && !mbar_wait(&up_empty[u], ((cc >> 1) & 1) ^ 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t aaddr = smem_u32(sA), w13 = smem_u32(sW13 + c * 32768);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16) {
          const uint64_t ad = MODE == MODE_SEQ ? sdesc_sw128(aaddr + (k16 >> 2) * (kATile / 2) + (k16 & 3) * 32)
                                               : sdesc_noswz(aaddr + k16 * 256, 128, 2048);
          tc_mma(tbase + kColUp + u * 128, ad, sdesc_sw128(w13 + (k16 >> 2) * 16384 + (k16 & 3) * 32), id128,
                 k16 != 0);
        }
        tc_commit(&up_full[u]);
        if (c == kChunks - 1) tc_commit(a_empty);
        return true;
      };
      auto issue_down = [&](int cc) -> bool {
        const int i = cc / kChunks, c = cc % kChunks, h = cc & 1;
        if (c == 0 && i >= 1 && !mbar_wait(dn_empty, (i - 1) & 1, abort_flag, a.err)) return false;
        if (!mbar_wait(&hm_full[h], (cc >> 1) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t w2 = smem_u32(sW2 + c * 16384);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_ts(tbase + kColDown, tbase + kColHid + h * 32 + k * 8, sdesc_sw128(w2 + k * 32), id128, (c | k) != 0);
        tc_commit(&hm_empty[h]);
        if (c == kChunks - 1) {
          tc_commit(dn_full);
          // the weights may be replaced once this tile's MMAs are done, if the next tile needs another group
          const int tile = blockIdx.x + i * gridDim.x, next = tile + gridDim.x;
          if (MODE == MODE_SEQ && next < n_tiles && tile_info<MODE>(a, next).g != tile_info<MODE>(a, tile).g)
            tc_commit(w_empty);
        }
        return true;
      };
      // Up projections run up to two chunks ahead of the down projections within a tile; at a tile boundary
      // all down projections of the current tile are issued before the next tile's first up projection.
      int nu = 0, nd = 0;
      while (ok && nd < total) {
        if (nu < total && nu <= nd + 2) {
          if (nu > 0 && nu % kChunks == 0 && nd < nu) {
            // finish the current tile's down projections first: the next tile's up projection may wait for
            // its activation load (or, for a sequence tile of another group, for the weight reload)
            ok = issue_down(nd++);
            continue;
          }
          ok = issue_up(nu++);
          continue;
        }
        ok = issue_down(nd++);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    const int q = warp & 3;               // TMEM lane quarter
    const int grp = (warp - 2) >> 2;      // column half
    const int rl = q * 32 + lane;         // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    bool ok = true;
    int bias_group = -1;
    uint64_t gj2[4];  // RMSNorm gain of this thread's head j (TM): one load per kernel
    if (MODE == MODE_TM) {
      const float2* gain = reinterpret_cast<const float2*>(a.tm_gain + layer * kD + (rl & 15) * 8);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 g = __ldg(gain + e);
        gj2[e] = f2pack(g.x, g.y);
      }
    }
    pdl_wait();
    for (int i = 0; i < n_my && ok; ++i) {
      const TileInfo ti = tile_info<MODE>(a, blockIdx.x + i * gridDim.x);
      if (ti.g != bias_group) {  // stage this group's biases (TM: once)
        if (bias_group >= 0) epi_sync();
        const int wsel = MODE == MODE_SEQ ? ti.g : layer;
        const float* b13g = (MODE == MODE_SEQ ? a.seq_b13 : a.tm_b13) + wsel * 2 * kHid;
        const float* b2g = (MODE == MODE_SEQ ? a.seq_b2 : a.tm_b2) + wsel * kD;
        const int t = threadIdx.x - 64;
        for (int k = t; k < 2 * kHid; k += kEpiWarps * 32) sb13[k] = b13g[k];
        for (int k = t; k < kD; k += kEpiWarps * 32) sb2[k] = b2g[k];
        epi_sync();
        bias_group = ti.g;
      }
      // TM: prefetch the residual Z[b][t][8j..8j+8) of this thread's 8 output tokens
      uint4 zres[8];
      const int bl = rl >> 4, j = rl & 15;
      const int64_t bcand = ti.row0 / kT + bl;
      if (MODE == MODE_TM) {
        // unconditional loads (rows past the batch read the last candidate and are never stored), so nothing
        // consumes the registers before the final epilogue and the loads stay in flight across the chunks
        const int64_t bsrc = bcand < a.B ? bcand : a.B - 1;
#pragma unroll
        for (int tt = 0; tt < 8; ++tt)
          zres[tt] = __ldg(reinterpret_cast<const uint4*>(zin + bsrc * kYD + (grp * 8 + tt) * kD + j * 8));
      }
      for (int c = 0; c < kChunks; ++c) {
        const int cc = i * kChunks + c, u = cc & 1;
        uint32_t ra[32], rg[32];
        ok = mbar_wait(&up_full[u], (cc >> 1) & 1, abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        tmem_ld32_nowait(tbase + lane_off + kColUp + u * 128 + grp * 32, ra);
        tmem_ld32_nowait(tbase + lane_off + kColUp + u * 128 + 64 + grp * 32, rg);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&up_empty[u]);
        const float* ba = sb13 + c * 128 + grp * 32;
        const float* bg = ba + 64;
        uint32_t hp[16];
        const float2* ba2 = reinterpret_cast<const float2*>(ba);
        const float2* bg2 = reinterpret_cast<const float2*>(bg);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 bav = ba2[e], bgv = bg2[e];
          const uint64_t av = add_f32x2(f2pack(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1])),
                                        f2pack(bav.x, bav.y));
          const uint64_t gv = add_f32x2(f2pack(__uint_as_float(rg[2 * e]), __uint_as_float(rg[2 * e + 1])),
                                        f2pack(bgv.x, bgv.y));
          hp[e] = silu_mul_bf16x2(av, gv);
        }
        if (cc >= 2) ok = mbar_wait(&hm_empty[u], ((cc >> 1) & 1) ^ 1, abort_flag, a.err);
        if (!ok) break;
        tc_fence_after();
        tmem_st16(tbase + lane_off + kColHid + u * 32 + grp * 16, hp);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&hm_full[u]);
      }
      if (!ok) break;
      // ---- output epilogue of this tile: columns [64 grp, 64 grp + 64) of the down accumulator
      ok = mbar_wait(dn_full, i & 1, abort_flag, a.err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dacc = tbase + lane_off + kColDown + grp * 64;
      uint32_t rv[2][32];
      tmem_ld32_nowait(dacc, rv[0]);
      tmem_ld32_nowait(dacc + 32, rv[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dn_empty);
      if (MODE == MODE_SEQ) {
        const int64_t row = ti.row0 + rl;
        if (row < ti.rows_end) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float* bb = sb2 + grp * 64 + h * 32;
            uint4* dst = reinterpret_cast<uint4*>(a.H + row * kD + grp * 64 + h * 32);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              uint4 p;
              uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = jj * 8 + 2 * e;
                pp[e] = pack_bf16(__uint_as_float(rv[h][x]) + bb[x], __uint_as_float(rv[h][x + 1]) + bb[x + 1]);
              }
              dst[jj] = p;
            }
          }
        }
      } else {
        // this thread holds F(mixed row (b, j)); output token t of candidate b takes F[(b, j)][8t..8t+8) as
        // its head j (Revert), adds the residual Z[b][t][8j..8j+8) and is RMS-normalised over its 128 dims,
        // whose 16 heads live in the 16 lanes that share b. This warp handles tokens [8 grp, 8 grp + 8).
        const bool live = bcand < a.B;
        // x = F + b2 + Z for 8 tokens x 8 dims (packed pairs), then the 8 sums of squares reduce together
        uint64_t x2[8][4];
        float ss[8];
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
          const int t = grp * 8 + tt;
          const float2* bb = reinterpret_cast<const float2*>(sb2 + t * 8);
          const __nv_bfloat162* zp = reinterpret_cast<const __nv_bfloat162*>(&zres[tt]);
          const uint32_t* v = &rv[tt >> 2][(tt & 3) * 8];
          uint64_t acc = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 b = bb[e];
            const float2 z = __bfloat1622float2(zp[e]);
            uint64_t xv = add_f32x2(f2pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), f2pack(b.x, b.y));
            xv = add_f32x2(xv, f2pack(z.x, z.y));
            x2[tt][e] = xv;
            acc = e == 0 ? mul_f32x2(xv, xv) : fma_f32x2(xv, xv, acc);
          }
          ss[tt] = __uint_as_float((uint32_t)acc) + __uint_as_float((uint32_t)(acc >> 32));
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) ss[tt] += __shfl_xor_sync(0xffffffffu, ss[tt], o);
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
          const float inv = rsqrtf(ss[tt] * (1.f / kD) + a.eps);
          const uint64_t inv2 = f2pack(inv, inv);
          uint4 p;
          uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint64_t y = mul_f32x2(mul_f32x2(x2[tt][e], inv2), gj2[e]);
            pp[e] = pack_bf16(__uint_as_float((uint32_t)y), __uint_as_float((uint32_t)(y >> 32)));
          }
          if (live) *reinterpret_cast<uint4*>(yout + bcand * kYD + (grp * 8 + tt) * kD + j * 8) = p;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

cudaError_t prepare_mlp_kernels() {
  cudaError_t e = cudaFuncSetAttribute(swiglu_mlp_kernel<MODE_SEQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(swiglu_mlp_kernel<MODE_TM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

cudaError_t launch_seq_mlp(const FwdArgs& a, const CUtensorMap& tmXs, const CUtensorMap& tmW13, const CUtensorMap& tmW2,
                           int n_tiles, cudaStream_t s) {
  const int grid = n_tiles < a.num_sms ? n_tiles : a.num_sms;
  return launch_kernel(swiglu_mlp_kernel<MODE_SEQ>, dim3(grid), dim3(kThreads), kSmemBytes, s, a.pdl != 0, a, tmXs,
                       tmW13, tmW2, 0, n_tiles, (const __nv_bfloat16*)nullptr, (__nv_bfloat16*)nullptr);
}

cudaError_t launch_tm_mlp(const FwdArgs& a, int layer, const __nv_bfloat16* zin, __nv_bfloat16* yout,
                          const CUtensorMap& tmZ, const CUtensorMap& tmW13, const CUtensorMap& tmW2, cudaStream_t s) {
  const int n_tiles = (a.B + 7) / 8;  // 8 candidates x 16 mixed rows per tile
  const int grid = n_tiles < a.num_sms ? n_tiles : a.num_sms;
  return launch_kernel(swiglu_mlp_kernel<MODE_TM>, dim3(grid), dim3(kThreads), kSmemBytes, s, a.pdl != 0, a, tmZ, tmW13,
                       tmW2, layer, n_tiles, zin, yout);
}

}  // namespace cvr
