// The user half of the tokeniser, once per request (iQIYI ad-CVR article 3.4.5: the user side is computed
// once and repeated lazily): xu[r][n] = tok_b[n] + sum_k Wtok_u[n][k] * U[r][k] for all 2048 packed tokeniser
// rows (the 13 tokens, then the first layer's query weights folded into the tokeniser). It runs as extra CTAs
// of the sequence-encoder launch, next to the encoder tiles, since it needs only the pooled user embeddings.
#pragma once
#include "cvr_internal.cuh"

namespace cvr {

constexpr int kXuCols = 32;                  // tokeniser rows per CTA
constexpr int kXuBlocks = kTokN / kXuCols;   // 64 CTAs
constexpr int kXuThreads = 512;              // threads taking part (named barrier 2)
constexpr int kXuReq = kXuThreads / 32;      // requests per pass: one per warp
constexpr int kXuWStride = kXuCols + 2;      // bf16 elements per staged k-row (conflict-free column reads)
constexpr int kXuSmemBytes = kUD * kXuWStride * 2 + kXuReq * kUD * 4;

__device__ __forceinline__ void xu_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kXuThreads) : "memory"); }

// Rows [32 blk, 32 blk + 32): the weight slice is staged transposed in shared memory (its loads are issued
// before waiting for the previous kernel), then the users kXuReq at a time; thread (row nn, request slot rs)
// finishes whole dot products with four independent partial sums.
__device__ __forceinline__ void xu_block(const FwdArgs& a, int blk, uint8_t* smem) {
  const int tid = threadIdx.x;
  if (tid >= kXuThreads) {
    pdl_wait();
    return;
  }
  __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(smem);                  // [256][34]: w[k][nn]
  float* act = reinterpret_cast<float*>(smem + kUD * kXuWStride * 2);         // [16][256]
  const int n0 = blk * kXuCols;
  // 32 rows x 256 bf16 = 1024 16-byte vectors: 2 per thread
  uint4 raw[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int v = tid + t * kXuThreads, nn = v >> 5, k8 = v & 31;
    raw[t] = __ldg(reinterpret_cast<const uint4*>(a.tokU + (int64_t)(n0 + nn) * kUD) + k8);
  }
  const int nn = tid & (kXuCols - 1), rs = tid >> 5;
  const float bias = __ldg(a.tok_b + n0 + nn);
  // warm L2 with the mean-pool query weights, which the column-sum kernel reads next
  {
    const int64_t lines = (int64_t)a.n_layers * kG * kD * kD * 2 / 128;
    const int64_t line = (int64_t)blk * kXuThreads + tid;
    if (line < lines) asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(a.qm) + line * 128));
  }
  pdl_wait();  // U comes from the sparse kernel
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int v = tid + t * kXuThreads, n = v >> 5, k8 = v & 31;
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[t]);
#pragma unroll
    for (int q = 0; q < 8; ++q) w[(k8 * 8 + q) * kXuWStride + n] = e[q];
  }
  for (int r0 = 0; r0 < a.R; r0 += kXuReq) {
    const int nr = min(kXuReq, a.R - r0);
    xu_sync();
    for (int v = tid; v < nr * (kUD / 8); v += kXuThreads) {  // 16-byte vectors of U
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(a.U + (int64_t)r0 * kUD) + v);
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        act[v * 8 + 2 * q] = __low2float(e[q]);
        act[v * 8 + 2 * q + 1] = __high2float(e[q]);
      }
    }
    xu_sync();
    if (rs < nr) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float* x = act + rs * kUD;
#pragma unroll 4
      for (int k = 0; k < kUD; k += 4) {
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[p] += __bfloat162float(w[(k + p) * kXuWStride + nn]) * x[k + p];
      }
      a.xu[(int64_t)(r0 + rs) * kTokN + n0 + nn] = (acc[0] + acc[1]) + (acc[2] + acc[3]) + bias;
    }
  }
}

}  // namespace cvr
