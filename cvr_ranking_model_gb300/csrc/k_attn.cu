// Query Decoding cross-attention (iQIYI ad-CVR article, section 3.2.3): for every candidate and group g,
// the group's query (4 heads of 32) attends over that request's encoded sequence H_g, which serves as
// both K and V; logits are scaled by 1/(tau*sqrt(32)) and normalised by a softmax over the sequence.
//
// One CTA = one group x 64 consecutive candidates (4 warps x 16). The request's K/V rows are staged once
// per CTA in shared memory in chunks of 64 positions (cp.async, double-buffered) and shared by all 64
// candidates; logits and P.V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with an online softmax
// across chunks, so any sequence length works with 35 KB of shared memory. The decoded tokens are
// written straight into slots 13..15 of the Token Mixer input.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kCandPerCta = 64;
constexpr int kChunk = 64;
constexpr int kKStride = kD + 8;  // padded smem row (272 B): conflict-free fragment loads

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__global__ void __launch_bounds__(128) attention_kernel(const __grid_constant__ FwdArgs a,
                                                        __nv_bfloat16* __restrict__ zin) {
  __shared__ __align__(16) __nv_bfloat16 Ks[2][kChunk][kKStride];
  const int g = blockIdx.y;
  const int b0 = blockIdx.x * kCandPerCta;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int L = a.L[g];
  const int R = a.R, B = a.B;
  pdl_trigger();
  pdl_wait();
  const int b_last = min(b0 + kCandPerCta, B) - 1;
  // request ids are validated by the sparse kernel; here they are only kept in range
  const int r_first = min(max(a.req_ids[b0], 0), R - 1);
  const int r_last = min(max(a.req_ids[b_last], 0), R - 1);

  const int rowA = b0 + warp * 16 + gid, rowB = rowA + 8;
  const int reqA = rowA < B ? a.req_ids[rowA] : -1;
  const int reqB = rowB < B ? a.req_ids[rowB] : -1;

  // query fragments (A operand, rows = candidates), 4 heads x 2 k-steps of 16
  // rows past the batch load the last candidate's query (their results are never stored): unconditional
  // loads keep all 32 in flight together
  uint32_t qf[kHeads][2][4];
  const int64_t qrA = min(rowA, B - 1), qrB = min(rowB, B - 1);
#pragma unroll
  for (int h = 0; h < kHeads; ++h)
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int col = g * kD + h * kHD + ks * 16 + 2 * tig;
      const uint32_t* qa = reinterpret_cast<const uint32_t*>(a.Q + qrA * (kG * kD) + col);
      const uint32_t* qb = reinterpret_cast<const uint32_t*>(a.Q + qrB * (kG * kD) + col);
      qf[h][ks][0] = __ldg(qa);
      qf[h][ks][1] = __ldg(qb);
      qf[h][ks][2] = __ldg(qa + 4);
      qf[h][ks][3] = __ldg(qb + 4);
    }
  // logits * log2(e) / (tau * sqrt(head_dim)) so that the softmax runs on exp2
  const float sl2 = 1.4426950408889634f / (a.tau * sqrtf((float)kHD));
  const int nchunks = (L + kChunk - 1) / kChunk;

  for (int r = r_first; r <= r_last; ++r) {
    const bool active = __any_sync(0xffffffffu, reqA == r || reqB == r);
    const __nv_bfloat16* Hb = a.H + (a.goff[g] + (int64_t)r * L) * kD;
    auto load_chunk = [&](int ch, int buf) {
      for (int i = threadIdx.x; i < kChunk * (kD / 8); i += blockDim.x) {
        const int row = i >> 4, c16 = i & 15;
        const int l = ch * kChunk + row;
        const bool ok = l < L;
        cp_async16(&Ks[buf][row][c16 * 8], Hb + (int64_t)(ok ? l : 0) * kD + c16 * 8, ok ? 16 : 0);
      }
    };
    float o[kHeads][4][4];
    float mx[kHeads][2], ls[kHeads][2];
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      mx[h][0] = mx[h][1] = -INFINITY;
      ls[h][0] = ls[h][1] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[h][j][i] = 0.f;
    }
    load_chunk(0, 0);
    cp_async_commit();
    for (int ch = 0; ch < nchunks; ++ch) {
      if (ch + 1 < nchunks) load_chunk(ch + 1, (ch + 1) & 1);
      cp_async_commit();
      cp_async_wait1();
      __syncthreads();
      if (active) {
        const int buf = ch & 1;
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          float s[8][4];
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const __nv_bfloat16* kp = &Ks[buf][nt * 8 + gid][h * kHD + ks * 16 + 2 * tig];
              const uint32_t kb0 = *reinterpret_cast<const uint32_t*>(kp);
              const uint32_t kb1 = *reinterpret_cast<const uint32_t*>(kp + 8);
              mma_bf16_16816(s[nt], qf[h][ks], kb0, kb1);
            }
          }
          float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int key = ch * kChunk + nt * 8 + 2 * tig + (i & 1);
              s[nt][i] = key < L ? s[nt][i] * sl2 : -INFINITY;
              if (i < 2)
                mA = fmaxf(mA, s[nt][i]);
              else
                mB = fmaxf(mB, s[nt][i]);
            }
          mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 1));
          mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, 2));
          mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 1));
          mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, 2));
          const float nA = fmaxf(mx[h][0], mA), nB = fmaxf(mx[h][1], mB);
          const float cA = exp2f(mx[h][0] - nA), cB = exp2f(mx[h][1] - nB);
          mx[h][0] = nA;
          mx[h][1] = nB;
          float sumA = 0.f, sumB = 0.f;
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - nA);
            s[nt][1] = exp2f(s[nt][1] - nA);
            s[nt][2] = exp2f(s[nt][2] - nB);
            s[nt][3] = exp2f(s[nt][3] - nB);
            sumA += s[nt][0] + s[nt][1];
            sumB += s[nt][2] + s[nt][3];
          }
          ls[h][0] = ls[h][0] * cA + sumA;
          ls[h][1] = ls[h][1] * cB + sumB;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[h][j][0] *= cA;
            o[h][j][1] *= cA;
            o[h][j][2] *= cB;
            o[h][j][3] *= cB;
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int ntp = 0; ntp < 2; ++ntp) {
              const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
              const int dim = h * kHD + ntp * 16 + (lane >> 4) * 8;
              uint32_t vb[4];
              ldmatrix_x4_trans(vb, &Ks[buf][key][dim]);
              mma_bf16_16816(o[h][2 * ntp], pa, vb[0], vb[1]);
              mma_bf16_16816(o[h][2 * ntp + 1], pa, vb[2], vb[3]);
            }
          }
        }
      }
      __syncthreads();
    }
    if (active) {
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        float lA = ls[h][0], lB = ls[h][1];
        lA += __shfl_xor_sync(0xffffffffu, lA, 1);
        lA += __shfl_xor_sync(0xffffffffu, lA, 2);
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
        const float iA = 1.f / lA, iB = 1.f / lB;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = kXD + g * kD + h * kHD + j * 8 + 2 * tig;
          if (reqA == r)
            *reinterpret_cast<uint32_t*>(zin + (int64_t)rowA * kYD + col) = pack_bf16(o[h][j][0] * iA, o[h][j][1] * iA);
          if (reqB == r)
            *reinterpret_cast<uint32_t*>(zin + (int64_t)rowB * kYD + col) = pack_bf16(o[h][j][2] * iB, o[h][j][3] * iB);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_attention(const FwdArgs& a, __nv_bfloat16* zin, cudaStream_t s) {
  const int nblk = (a.B + kCandPerCta - 1) / kCandPerCta;
  return launch_kernel(attention_kernel, dim3(nblk, kG), dim3(128), 0, s, a.pdl != 0, a, zin);
}

}  // namespace cvr
