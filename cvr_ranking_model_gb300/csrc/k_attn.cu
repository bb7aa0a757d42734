// Query Decoding cross-attention (iQIYI ad-CVR article, section 3.2.3): for every candidate and group g,
// the group's query (4 heads of 32) attends over that request's encoded sequence H_g, which serves as
// both K and V; logits are scaled by 1/(tau*sqrt(32)) and normalised by a softmax over the sequence.
//
// One CTA = one group x 32 consecutive candidates (two m16 MMA tiles), 8 warps: warp w owns candidate tile
// w / 4 and head w % 4 for the whole sequence, so its online-softmax state never needs merging. All warps
// share the K/V chunks of 64 positions, staged by the whole CTA with cp.async into a double buffer; every
// K/V row is read once per 32 candidates. Logits and P.V run on mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with the softmax on exp2, and the decoded tokens are written straight into slots 13..15 of
// the Token Mixer input.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kCandPerCta = 32;
constexpr int kWarps = 8;
constexpr int kChunk = 64;                        // positions per step
constexpr int kKStride = kD + 8;                  // padded smem row (272 B): conflict-free fragment loads
constexpr int kBufBytes = kChunk * kKStride * 2;  // 17408 B
constexpr int kSmemBytes = 2 * kBufBytes;         // 34816 B

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
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kWarps * 32) attention_kernel(const __grid_constant__ FwdArgs a,
                                                                __nv_bfloat16* __restrict__ zin) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int g = blockIdx.y;
  const int b0 = blockIdx.x * kCandPerCta;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int mt = warp >> 2, h = warp & 3;  // candidate tile and head of this warp
  const int L = a.L[g];
  const int R = a.R, B = a.B;
  __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(smem);  // 2 chunks of [64][136]
  pdl_trigger();
  pdl_wait();
  const int b_last = min(b0 + kCandPerCta, B) - 1;
  // request ids are validated by the sparse kernel; here they are only kept in range
  const int r_first = min(max(a.req_ids[b0], 0), R - 1);
  const int r_last = min(max(a.req_ids[b_last], 0), R - 1);
  const int rowA = b0 + mt * 16 + gid, rowB = rowA + 8;
  const int reqA = rowA < B ? a.req_ids[rowA] : -1;
  const int reqB = rowB < B ? a.req_ids[rowB] : -1;

  // query fragments of head h (A operand, rows = candidates); rows past the batch load the last candidate's
  // query (never stored), so all loads are unconditional and in flight together
  uint32_t qf[2][4];
  const int64_t qrA = min(rowA, B - 1), qrB = min(rowB, B - 1);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int col = g * kD + h * kHD + ks * 16 + 2 * tig;
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(a.Q + qrA * (kG * kD) + col);
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(a.Q + qrB * (kG * kD) + col);
    qf[ks][0] = __ldg(qa);
    qf[ks][1] = __ldg(qb);
    qf[ks][2] = __ldg(qa + 4);
    qf[ks][3] = __ldg(qb + 4);
  }
  // logits * log2(e) / (tau * sqrt(head_dim)) so that the softmax runs on exp2
  const float sl2 = 1.4426950408889634f / (a.tau * sqrtf((float)kHD));

  for (int r = r_first; r <= r_last; ++r) {
    const __nv_bfloat16* Hb = a.H + (a.goff[g] + (int64_t)r * L) * kD;
    // keys: the request's real events (variable-length sequences mask the padding out); none -> zero token
    const int Lr = seq_len_of(a, r, g);
    const int nchunks = (Lr + kChunk - 1) / kChunk;
    // one chunk = 64 rows x 16 pieces of 16 bytes, 4 per thread; rows past L are zero-filled
    auto load_chunk = [&](int ch, int slot) {
      __nv_bfloat16* dst = buf + slot * (kChunk * kKStride);
#pragma unroll
      for (int i = 0; i < kChunk * (kD / 8) / (kWarps * 32); ++i) {
        const int v = tid + i * kWarps * 32, row = v >> 4, c16 = v & 15;
        const int l = ch * kChunk + row;
        const bool ok = l < Lr;
        cp_async16(dst + row * kKStride + c16 * 8, Hb + (int64_t)(ok ? l : 0) * kD + c16 * 8, ok ? 16 : 0);
      }
    };
    float o[4][4];
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] = 0.f;
    __syncthreads();  // the previous request's chunks have been read by every warp
    if (nchunks > 0) load_chunk(0, 0);
    cp_async_commit();
    for (int ch = 0; ch < nchunks; ++ch) {
      if (ch + 1 < nchunks) load_chunk(ch + 1, (ch + 1) & 1);
      cp_async_commit();
      cp_async_wait1();
      __syncthreads();  // chunk ch has landed for every warp
      const __nv_bfloat16* Ks = buf + (ch & 1) * (kChunk * kKStride);
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const __nv_bfloat16* kp = Ks + (nt * 8 + gid) * kKStride + h * kHD + ks * 16 + 2 * tig;
          mma_bf16_16816(s[nt], qf[ks], *reinterpret_cast<const uint32_t*>(kp),
                         *reinterpret_cast<const uint32_t*>(kp + 8));
        }
      }
      float cA = -INFINITY, cB = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = ch * kChunk + nt * 8 + 2 * tig + (i & 1);
          s[nt][i] = key < Lr ? s[nt][i] * sl2 : -INFINITY;
          if (i < 2)
            cA = fmaxf(cA, s[nt][i]);
          else
            cB = fmaxf(cB, s[nt][i]);
        }
      cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 1));
      cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 2));
      cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 1));
      cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 2));
      const float nA = fmaxf(mA, cA), nB = fmaxf(mB, cB);
      const float fA = ex2(mA - nA), fB = ex2(mB - nB);
      mA = nA;
      mB = nB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = ex2(s[nt][0] - nA);
        s[nt][1] = ex2(s[nt][1] - nA);
        s[nt][2] = ex2(s[nt][2] - nB);
        s[nt][3] = ex2(s[nt][3] - nB);
        sumA += s[nt][0] + s[nt][1];
        sumB += s[nt][2] + s[nt][3];
      }
      lA = lA * fA + sumA;
      lB = lB * fB + sumB;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[j][0] *= fA;
        o[j][1] *= fA;
        o[j][2] *= fB;
        o[j][3] *= fB;
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
          ldmatrix_x4_trans(vb, Ks + key * kKStride + dim);
          mma_bf16_16816(o[2 * ntp], pa, vb[0], vb[1]);
          mma_bf16_16816(o[2 * ntp + 1], pa, vb[2], vb[3]);
        }
      }
      __syncthreads();  // every warp is done with chunk ch before it is refilled
    }
    // row sums over the 4 threads of a row, then the decoded token of head h
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const float iA = Lr > 0 ? 1.f / lA : 0.f, iB = Lr > 0 ? 1.f / lB : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = kXD + g * kD + h * kHD + j * 8 + 2 * tig;
      if (reqA == r)
        *reinterpret_cast<uint32_t*>(zin + (int64_t)rowA * kYD + col) = pack_bf16(o[j][0] * iA, o[j][1] * iA);
      if (reqB == r)
        *reinterpret_cast<uint32_t*>(zin + (int64_t)rowB * kYD + col) = pack_bf16(o[j][2] * iB, o[j][3] * iB);
    }
  }
}

}  // namespace

cudaError_t prepare_attention_kernel() {
  return cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_attention(const FwdArgs& a, __nv_bfloat16* zin, cudaStream_t s) {
  const int nblk = (a.B + kCandPerCta - 1) / kCandPerCta;
  return launch_kernel(attention_kernel, dim3(nblk, kG), dim3(kWarps * 32), kSmemBytes, s, a.pdl != 0, a, zin);
}

}  // namespace cvr
