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
// One CTA = 128 rows. The up projection runs as two N=256 MMAs (W1 and W3 rows interleaved per 128
// hidden units) into the whole 512-column TMEM; the epilogue warps turn each half into silu(a)*b and
// write the bf16 hidden tile into 128B-swizzled shared memory, which is the A operand of the down
// projection (N=128, accumulated into TMEM columns 0..127). The hidden activations never leave the SM.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kThreads = 192;
constexpr int kATileBytes = 128 * kD * 2;       // 32 KB
constexpr int kWBufBytes = 256 * kD * 2;        // 64 KB
constexpr int kHTileBytes = 128 * kHid * 2;     // 64 KB
constexpr int kOffA = 0;
constexpr int kOffW0 = kOffA + kATileBytes;
constexpr int kOffW1 = kOffW0 + kWBufBytes;
constexpr int kOffH = kOffW1 + kWBufBytes;
constexpr int kOffBar = kOffH + kHTileBytes;
constexpr int kSmemBytes = 1024 + kOffBar + 128;

enum { MODE_SEQ = 0, MODE_TM = 1 };

__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    swiglu_mlp_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2, int layer,
                      const __nv_bfloat16* __restrict__ zin, __nv_bfloat16* __restrict__ yout) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + kOffA;
  uint8_t* sW0 = smem + kOffW0;
  uint8_t* sW1 = smem + kOffW1;
  uint8_t* sH = smem + kOffH;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* barA = bars + 0;
  uint64_t* barW0 = bars + 1;
  uint64_t* barW1 = bars + 2;
  uint64_t* barW2 = bars + 3;
  uint64_t* barUp0 = bars + 4;
  uint64_t* barUp1 = bars + 5;
  uint64_t* barHm = bars + 6;
  uint64_t* barDown = bars + 7;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile -> rows
  int g = 0;
  int64_t row0 = 0;      // first A row of the tile (SEQ: row in the grouped layout; TM: mixed row 16*b + j)
  int64_t rows_end = 0;  // rows of this tile's problem
  int w13_row = 0, w2_row = 0;
  if (MODE == MODE_SEQ) {
    int tile = blockIdx.x;
    while (g < kG - 1) {
      const int tg = (int)(((int64_t)a.R * a.L[g] + 127) / 128);
      if (tile < tg) break;
      tile -= tg;
      ++g;
    }
    row0 = a.goff[g] + (int64_t)tile * 128;
    rows_end = a.goff[g] + (int64_t)a.R * a.L[g];
    w13_row = g * 2 * kHid;
    w2_row = g * kD;
  } else {
    row0 = (int64_t)blockIdx.x * 128;
    rows_end = (int64_t)a.B * kT;
    w13_row = layer * 2 * kHid;
    w2_row = layer * kD;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&bars[i], i == 6 ? 128 : 1);
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

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(barA, kATileBytes);
      if (MODE == MODE_SEQ) {
        tma_load_2d(sA, &tmA, barA, 0, (int)row0);
        tma_load_2d(sA + kATileBytes / 2, &tmA, barA, 64, (int)row0);
      } else {
        // Z[b][t][8j+e] -> smem [b][j/8][t][j%8][e]: core matrices of 8 mixed rows x 8 K-elements
        tma_load_5d(sA, &tmA, barA, 0, 0, 0, 0, (int)(row0 / kT));
      }
      mbar_expect_tx(barW0, kWBufBytes);
      tma_load_2d(sW0, &tmW13, barW0, 0, w13_row);
      tma_load_2d(sW0 + kWBufBytes / 2, &tmW13, barW0, 64, w13_row);
      mbar_expect_tx(barW1, kWBufBytes);
      tma_load_2d(sW1, &tmW13, barW1, 0, w13_row + kHid);
      tma_load_2d(sW1 + kWBufBytes / 2, &tmW13, barW1, 64, w13_row + kHid);
      if (mbar_wait(barUp0, 0, abort_flag, a.err)) {  // the up-0 MMAs have finished reading buffer 0
        mbar_expect_tx(barW2, kWBufBytes);
        for (int kb = 0; kb < 4; ++kb) tma_load_2d(sW0 + kb * (kWBufBytes / 4), &tmW2, barW2, kb * 64, w2_row);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id256 = idesc_bf16(128, 256);
      constexpr uint32_t id128 = idesc_bf16(128, 128);
      auto adesc = [&](int k16) -> uint64_t {
        if (MODE == MODE_SEQ) return sdesc_sw128(smem_u32(sA) + (k16 >> 2) * (kATileBytes / 2) + (k16 & 3) * 32);
        return sdesc_noswz(smem_u32(sA) + k16 * 256, 128, 2048);
      };
      bool ok = mbar_wait(barA, 0, abort_flag, a.err) && mbar_wait(barW0, 0, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        for (int k16 = 0; k16 < kD / 16; ++k16)
          tc_mma(tbase, adesc(k16), sdesc_sw128(smem_u32(sW0) + (k16 >> 2) * (kWBufBytes / 2) + (k16 & 3) * 32), id256,
                 k16 != 0);
        tc_commit(barUp0);
        ok = mbar_wait(barW1, 0, abort_flag, a.err);
      }
      if (ok) {
        tc_fence_after();
        for (int k16 = 0; k16 < kD / 16; ++k16)
          tc_mma(tbase + 256, adesc(k16), sdesc_sw128(smem_u32(sW1) + (k16 >> 2) * (kWBufBytes / 2) + (k16 & 3) * 32),
                 id256, k16 != 0);
        tc_commit(barUp1);
        ok = mbar_wait(barHm, 0, abort_flag, a.err) && mbar_wait(barW2, 0, abort_flag, a.err);
      }
      if (ok) {
        tc_fence_after();
        for (int k16 = 0; k16 < kHid / 16; ++k16)
          tc_mma(tbase, sdesc_sw128(smem_u32(sH) + (k16 >> 2) * (kHTileBytes / 4) + (k16 & 3) * 32),
                 sdesc_sw128(smem_u32(sW0) + (k16 >> 2) * (kWBufBytes / 4) + (k16 & 3) * 32), id128, k16 != 0);
        tc_commit(barDown);
      }
    }
  } else {
    const int q = warp & 3;
    const int rl = q * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float* b13 = (MODE == MODE_SEQ ? a.seq_b13 + g * 2 * kHid : a.tm_b13 + layer * 2 * kHid);
    // ---- hidden = silu(W1 x + b1) * (W3 x + b3), written as the bf16 A operand of the down projection
    bool ok = true;
    for (int h = 0; h < 2 && ok; ++h) {
      ok = mbar_wait(h == 0 ? barUp0 : barUp1, 0, abort_flag, a.err);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float va[32], vg[32], ba[32], bg[32];
        ldg32(b13 + h * 256 + c * 32, ba);
        ldg32(b13 + h * 256 + 128 + c * 32, bg);
        tmem_ld32(tbase + lane_off + h * 256 + c * 32, va);
        tmem_ld32(tbase + lane_off + h * 256 + 128 + c * 32, vg);
        const int kb = h * 2 + (c >> 1);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint4 p;
          uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = jj * 8 + 2 * i;
            pp[i] = pack_bf16(silu(va[j] + ba[j]) * (vg[j] + bg[j]), silu(va[j + 1] + ba[j + 1]) * (vg[j + 1] + bg[j + 1]));
          }
          *reinterpret_cast<uint4*>(sH + kb * (kHTileBytes / 4) + sw128_offset(rl, (c & 1) * 4 + jj)) = p;
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(barHm);
    // ---- output epilogue
    if (ok && mbar_wait(barDown, 0, abort_flag, a.err)) {
      tc_fence_after();
      const int64_t row = row0 + rl;
      if (MODE == MODE_SEQ) {
        const float* b2 = a.seq_b2 + g * kD;
        const bool live = row < rows_end;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32], bb[32];
          ldg32(b2 + c * 32, bb);
          tmem_ld32(tbase + lane_off + c * 32, v);
          if (!live) continue;
          uint4* dst = reinterpret_cast<uint4*>(a.H + row * kD + c * 32);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint4 p;
            uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = jj * 8 + 2 * i;
              pp[i] = pack_bf16(v[j] + bb[j], v[j + 1] + bb[j + 1]);
            }
            dst[jj] = p;
          }
        }
      } else {
        // this thread holds F(mixed row (b, j)); output token t of candidate b takes F[(b, j)][8t..8t+8) as
        // its head j (Revert), adds the residual Z[b][t][8j..8j+8) and is RMS-normalised over its 128 dims,
        // whose 16 heads live in the 16 lanes that share b.
        const float* b2 = a.tm_b2 + layer * kD;
        const float* gain = a.tm_gain + layer * kD;
        const int bl = rl >> 4, j = rl & 15, jhi = j >> 3, jlo = j & 7;
        const int64_t b = row0 / kT + bl;
        const bool live = b < a.B;
        float gj[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) gj[e] = gain[j * 8 + e];
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32], bb[32];
          ldg32(b2 + c * 32, bb);
          tmem_ld32(tbase + lane_off + c * 32, v);
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const int t = c * 4 + tt;
            const uint4 zr = *reinterpret_cast<const uint4*>(sA + ((((bl * 2 + jhi) * kT + t) * 8 + jlo) * 16));
            const __nv_bfloat162* zp = reinterpret_cast<const __nv_bfloat162*>(&zr);
            float x[8];
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              x[2 * i] = v[tt * 8 + 2 * i] + bb[tt * 8 + 2 * i] + __low2float(zp[i]);
              x[2 * i + 1] = v[tt * 8 + 2 * i + 1] + bb[tt * 8 + 2 * i + 1] + __high2float(zp[i]);
              ss += x[2 * i] * x[2 * i] + x[2 * i + 1] * x[2 * i + 1];
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            const float inv = rsqrtf(ss * (1.f / kD) + a.eps);
            if (live) {
              uint4 p;
              uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                pp[i] = pack_bf16(x[2 * i] * inv * gj[2 * i], x[2 * i + 1] * inv * gj[2 * i + 1]);
              *reinterpret_cast<uint4*>(yout + b * kYD + t * kD + j * 8) = p;
            }
          }
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
  swiglu_mlp_kernel<MODE_SEQ><<<n_tiles, kThreads, kSmemBytes, s>>>(a, tmXs, tmW13, tmW2, 0, nullptr, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_tm_mlp(const FwdArgs& a, int layer, const __nv_bfloat16* zin, __nv_bfloat16* yout,
                          const CUtensorMap& tmZ, const CUtensorMap& tmW13, const CUtensorMap& tmW2, cudaStream_t s) {
  const int n_tiles = (a.B + 7) / 8;  // 8 candidates x 16 mixed rows per tile
  swiglu_mlp_kernel<MODE_TM><<<n_tiles, kThreads, kSmemBytes, s>>>(a, tmZ, tmW13, tmW2, layer, zin, yout);
  return cudaGetLastError();
}

}  // namespace cvr
