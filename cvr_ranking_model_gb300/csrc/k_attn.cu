// Query Decoding cross-attention (iQIYI ad-CVR article, section 3.2.3): for every candidate and group g,
// the group's query (4 heads of 32) attends over that request's encoded sequence H_g, which serves as
// both K and V; logits are scaled by 1/(tau*sqrt(32)) and normalised by a softmax over the sequence.
//
// One CTA = one group x 16 consecutive candidates (one m16 MMA tile), 4 warps. The warps split the sequence:
// warp w takes chunks w, w+4, w+8, ... of 32 positions, each staged by cp.async into the warp's own
// double buffer, so every K/V row is read once per 16 candidates and the warps never wait on each other.
// Logits and P.V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with an online softmax; the four
// partial (max, sum, P.V) states are then merged through shared memory, warp h finishing head h, and the
// decoded tokens are written straight into slots 13..15 of the Token Mixer input.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kCandPerCta = 16;
constexpr int kWarps = 4;
constexpr int kChunk = 32;                       // positions per warp step
constexpr int kKStride = kD + 8;                 // padded smem row (272 B): conflict-free fragment loads
constexpr int kBufBytes = kChunk * kKStride * 2;  // 8704 B
constexpr int kStateFloats = 80;                 // per thread: max[4][2], sum[4][2], O[4][4][4]
constexpr int kSmemBytes = kWarps * 2 * kBufBytes;  // 69632 B (the merge state, 40 KB, reuses it)
static_assert(kWarps * kStateFloats * 32 * 4 <= kSmemBytes, "merge state fits in the chunk buffers");

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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int L = a.L[g];
  const int R = a.R, B = a.B;
  __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(smem + warp * 2 * kBufBytes);  // this warp's 2 chunks
  float* state = reinterpret_cast<float*>(smem);                                       // [warp][field][lane]
  pdl_trigger();
  pdl_wait();
  const int b_last = min(b0 + kCandPerCta, B) - 1;
  // request ids are validated by the sparse kernel; here they are only kept in range
  const int r_first = min(max(a.req_ids[b0], 0), R - 1);
  const int r_last = min(max(a.req_ids[b_last], 0), R - 1);
  const int rowA = b0 + gid, rowB = rowA + 8;
  const int reqA = rowA < B ? a.req_ids[rowA] : -1;
  const int reqB = rowB < B ? a.req_ids[rowB] : -1;

  // query fragments (A operand, rows = candidates); rows past the batch load the last candidate's query
  // (never stored), so all 32 loads are unconditional and in flight together
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
    const __nv_bfloat16* Hb = a.H + (a.goff[g] + (int64_t)r * L) * kD;
    auto load_chunk = [&](int ch, int slot) {
      __nv_bfloat16* dst = buf + slot * (kChunk * kKStride);
#pragma unroll
      for (int i = 0; i < kChunk * (kD / 8) / 32; ++i) {
        const int v = lane + i * 32, row = v >> 4, c16 = v & 15;
        const int l = ch * kChunk + row;
        const bool ok = l < L;
        cp_async16(dst + row * kKStride + c16 * 8, Hb + (int64_t)(ok ? l : 0) * kD + c16 * 8, ok ? 16 : 0);
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
    if (warp < nchunks) load_chunk(warp, 0);
    cp_async_commit();
    int k = 0;
    for (int ch = warp; ch < nchunks; ch += kWarps, ++k) {
      if (ch + kWarps < nchunks) load_chunk(ch + kWarps, (k + 1) & 1);
      cp_async_commit();
      cp_async_wait1();
      __syncwarp();
      const __nv_bfloat16* Ks = buf + (k & 1) * (kChunk * kKStride);
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        float s[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const __nv_bfloat16* kp = Ks + (nt * 8 + gid) * kKStride + h * kHD + ks * 16 + 2 * tig;
            mma_bf16_16816(s[nt], qf[h][ks], *reinterpret_cast<const uint32_t*>(kp),
                           *reinterpret_cast<const uint32_t*>(kp + 8));
          }
        }
        float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
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
        const float cA = ex2(mx[h][0] - nA), cB = ex2(mx[h][1] - nB);
        mx[h][0] = nA;
        mx[h][1] = nB;
        float sumA = 0.f, sumB = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          s[nt][0] = ex2(s[nt][0] - nA);
          s[nt][1] = ex2(s[nt][1] - nA);
          s[nt][2] = ex2(s[nt][2] - nB);
          s[nt][3] = ex2(s[nt][3] - nB);
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
        for (int kk = 0; kk < 2; ++kk) {
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
            mma_bf16_16816(o[h][2 * ntp], pa, vb[0], vb[1]);
            mma_bf16_16816(o[h][2 * ntp + 1], pa, vb[2], vb[3]);
          }
        }
      }
      __syncwarp();
    }
    // ---- merge the four warps' partial states; warp h finishes head h
    __syncthreads();  // every warp is done with its chunk buffers (the state overwrites them)
    {
      float* st = state + warp * kStateFloats * 32 + lane;
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        st[(h * 2 + 0) * 32] = mx[h][0];
        st[(h * 2 + 1) * 32] = mx[h][1];
        st[(8 + h * 2 + 0) * 32] = ls[h][0];
        st[(8 + h * 2 + 1) * 32] = ls[h][1];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) st[(16 + (h * 4 + j) * 4 + i) * 32] = o[h][j][i];
      }
    }
    __syncthreads();
    {
      const int h = warp;
      float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* st = state + w * kStateFloats * 32 + lane;
        m0 = fmaxf(m0, st[(h * 2 + 0) * 32]);
        m1 = fmaxf(m1, st[(h * 2 + 1) * 32]);
      }
      float l0 = 0.f, l1 = 0.f, acc[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* st = state + w * kStateFloats * 32 + lane;
        const float f0 = ex2(st[(h * 2 + 0) * 32] - m0), f1 = ex2(st[(h * 2 + 1) * 32] - m1);
        l0 += st[(8 + h * 2 + 0) * 32] * f0;
        l1 += st[(8 + h * 2 + 1) * 32] * f1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[j][0] += st[(16 + (h * 4 + j) * 4 + 0) * 32] * f0;
          acc[j][1] += st[(16 + (h * 4 + j) * 4 + 1) * 32] * f0;
          acc[j][2] += st[(16 + (h * 4 + j) * 4 + 2) * 32] * f1;
          acc[j][3] += st[(16 + (h * 4 + j) * 4 + 3) * 32] * f1;
        }
      }
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = kXD + g * kD + h * kHD + j * 8 + 2 * tig;
        if (reqA == r)
          *reinterpret_cast<uint32_t*>(zin + (int64_t)rowA * kYD + col) = pack_bf16(acc[j][0] * i0, acc[j][1] * i0);
        if (reqB == r)
          *reinterpret_cast<uint32_t*>(zin + (int64_t)rowB * kYD + col) = pack_bf16(acc[j][2] * i1, acc[j][3] * i1);
      }
    }
    __syncthreads();  // the state is read before the next request's chunks overwrite it
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
