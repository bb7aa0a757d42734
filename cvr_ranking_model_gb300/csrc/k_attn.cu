// Query Decoding cross-attention (iQIYI ad-CVR article, section 3.2.3): for every candidate and group g,
// the group's query (4 heads of 32) attends over that request's encoded sequence H_g, which serves as
// both K and V; logits are scaled by 1/(tau*sqrt(32)) and normalised by a softmax over the sequence.
//
// One CTA = one group x 32 consecutive candidates (two m16 MMA tiles), 8 warps: warp w owns candidate tile
// w / 4 and head w % 4 for the whole sequence, so its online-softmax state never needs merging within the
// CTA. A group longer than 512 positions is split over several CTAs (when the tile holds one request); the
// last of them to finish -- found with a counter, nobody waits -- merges their states. All warps
// share the K/V chunks of 64 positions, staged by the whole CTA with cp.async into a ring of 5 slots with
// 3 chunks in flight ahead of the one in use (a 200-position sequence is in flight at once); every K/V row
// is read once per 32 candidates. Logits and P.V run on mma.sync m16n8k16 (bf16 in, fp32
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
constexpr int kNBuf = 5;                          // ring slots
constexpr int kAhead = 3;                         // chunks in flight ahead of the one in use
constexpr int kSmemBytes = kNBuf * kBufBytes;     // 87040 B: two CTAs per SM
static_assert(kAhead <= kNBuf - 2, "a refilled slot was read two chunks ago, before the last barrier");
static_assert(kChunk == kAttnChunk, "split sizing uses the same chunk");

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
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kWarps * 32, 2) attention_kernel(const __grid_constant__ FwdArgs a,
                                                                __nv_bfloat16* __restrict__ zin) {
  extern __shared__ __align__(16) uint8_t smem[];
  CVR_TL_BEGIN(TL_ATTENTION);
  const int g = a.g_order[blockIdx.y], sp = blockIdx.z;
  const int b0 = blockIdx.x * kCandPerCta;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int mt = warp >> 2, h = warp & 3;  // candidate tile and head of this warp
  const int L = a.L[g];
  const int R = a.R, B = a.B;
  const int n_split = split_count(L);  // this group's splits of the sequence
  __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(smem);  // kNBuf chunks of [64][136]
  pdl_trigger();
  if (sp >= n_split) return;
  pdl_wait();
  if (threadIdx.x == 0) CVR_TL_WAITED();
  const int b_last = min(b0 + kCandPerCta, B) - 1;
  // request ids are validated by the sparse kernel; here they are only kept in range
  const int r_first = min(max(a.req_ids[b0], 0), R - 1);
  const int r_last = min(max(a.req_ids[b_last], 0), R - 1);
  // A long sequence is split over n_split CTAs when the tile holds one request; otherwise the first split's
  // CTA takes every position of every request of its tile.
  const bool split = n_split > 1 && r_first == r_last;
  if (!split && sp > 0) return;
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
  if (a.q_add) {
    // the first layer's queries still lack the mean-pooled sequence term of their request (the tokeniser ran
    // next to the sequence encoder): q = q + qb[r], rounded to bf16 again
    const int rA = min(max(a.req_ids[qrA], 0), R - 1), rB = min(max(a.req_ids[qrB], 0), R - 1);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int col = g * kD + h * kHD + ks * 16 + 2 * tig;
      const float2* pa = reinterpret_cast<const float2*>(a.qb + (int64_t)rA * (kG * kD) + col);
      const float2* pb = reinterpret_cast<const float2*>(a.qb + (int64_t)rB * (kG * kD) + col);
      const float2 ta0 = __ldg(pa), tb0 = __ldg(pb), ta1 = __ldg(pa + 4), tb1 = __ldg(pb + 4);
      auto add2 = [](uint32_t q, float2 t) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&q);
        return pack_bf16(__low2float(v) + t.x, __high2float(v) + t.y);
      };
      qf[ks][0] = add2(qf[ks][0], ta0);
      qf[ks][1] = add2(qf[ks][1], tb0);
      qf[ks][2] = add2(qf[ks][2], ta1);
      qf[ks][3] = add2(qf[ks][3], tb1);
    }
  }
  // logits * log2(e) / (tau * sqrt(head_dim)) so that the softmax runs on exp2
  const float sl2 = 1.4426950408889634f / (a.tau * sqrtf((float)kHD));

  // online-softmax state of this thread: rows A (gid) and B (gid + 8), 8 of head h's 32 output columns each
  float o[4][4];
  float mA, mB, lA, lB;
  // positions [64 c_begin, 64 c_end) of request r's group-g sequence, of which Lr are real events
  auto run_chunks = [&](int r, int Lr, int c_begin, int c_end) {
    const __nv_bfloat16* Hb = a.H + (a.goff[g] + (int64_t)r * L) * kD;
    // one chunk = 64 rows x 16 pieces of 16 bytes, 4 per thread; rows past Lr are zero-filled
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
    mA = mB = -INFINITY;
    lA = lB = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] = 0.f;
    cta_sync();  // the previous request's chunks have been read by every warp
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {  // (one commit group per chunk, empty past the last)
      if (c_begin + i < c_end) load_chunk(c_begin + i, i);
      cp_async_commit();
    }
    for (int ch = c_begin; ch < c_end; ++ch) {
      const int j = ch - c_begin, slot = j % kNBuf;
      // the slot of chunk ch - 2: every warp finished it before it met the barrier of chunk ch - 1
      if (ch + kAhead < c_end) load_chunk(ch + kAhead, (j + kAhead) % kNBuf);
      cp_async_commit();
      cp_async_wait<kAhead>();
      cta_sync();  // chunk ch has landed for every warp
      const __nv_bfloat16* Ks = buf + slot * (kChunk * kKStride);
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
      // the row maxima on the raw logits (the scale is positive); only the sequence's last chunk has keys to mask
      if ((ch + 1) * kChunk > Lr) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (ch * kChunk + nt * 8 + 2 * tig + (i & 1) >= Lr) s[nt][i] = -INFINITY;
      }
      float cA = -INFINITY, cB = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        cA = fmaxf(cA, fmaxf(s[nt][0], s[nt][1]));
        cB = fmaxf(cB, fmaxf(s[nt][2], s[nt][3]));
      }
      cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 1));
      cA = fmaxf(cA, __shfl_xor_sync(0xffffffffu, cA, 2));
      cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 1));
      cB = fmaxf(cB, __shfl_xor_sync(0xffffffffu, cB, 2));
      // running maxima in the scaled (log2) domain; p = 2^(s sl2 - m), the scale folded into one FMA per logit
      const float nA = fmaxf(mA, cA * sl2), nB = fmaxf(mB, cB * sl2);
      const float fA = ex2(mA - nA), fB = ex2(mB - nB);
      mA = nA;
      mB = nB;
      float sumA = 0.f, sumB = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = ex2(fmaf(s[nt][0], sl2, -nA));
        s[nt][1] = ex2(fmaf(s[nt][1], sl2, -nA));
        s[nt][2] = ex2(fmaf(s[nt][2], sl2, -nB));
        s[nt][3] = ex2(fmaf(s[nt][3], sl2, -nB));
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
    }
  };
  // row sums over the 4 threads of a row, then the decoded token of head h for the rows of request r
  auto finish = [&](int r, int Lr) {
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
  };

  // this group's tokens of the tile are written: count them for the Token Mixer, whose tiles of these candidates
  // start once every group is in (a CTA barrier, then one release at GPU scope covers all the CTA's writes)
  auto publish = [&]() {
    if (!a.attn_ready) return;
    cta_sync();
    if (tid == 0) red_release_add(a.attn_ready + blockIdx.x, 1u);
  };
  if (!split) {
    for (int r = r_first; r <= r_last; ++r) {
      // keys: the request's real events (variable-length sequences mask the padding out); none -> zero token
      const int Lr = seq_len_of(a, r, g);
      run_chunks(r, Lr, 0, (Lr + kChunk - 1) / kChunk);
      finish(r, Lr);
    }
    publish();
    return;
  }
  // ---- split: this CTA's positions, its state to the workspace, the last split of the tile merges them
  const int r = r_first;
  const int Lr = seq_len_of(a, r, g);
  const int nch = (Lr + kChunk - 1) / kChunk;
  const int per = ((L + kChunk - 1) / kChunk + n_split - 1) / n_split;  // chunks per split (of the padded length)
  run_chunks(r, Lr, min(sp * per, nch), min((sp + 1) * per, nch));
  const int64_t slot = (int64_t)blockIdx.x * kG + g;
  float4* st = reinterpret_cast<float4*>(a.attn_state) + ((slot * a.attn_splits + sp) * (kWarps * 32) + tid) * 5;
  st[0] = make_float4(mA, mB, lA, lB);
#pragma unroll
  for (int j = 0; j < 4; ++j) st[1 + j] = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
  __shared__ int last;
  __threadfence();
  cta_sync();
  if (tid == 0) last = atomicAdd(a.attn_count + slot, 1u) == (unsigned)(n_split - 1);
  cta_sync();
  if (!last) return;
  // merge in split order: M = max m_s, l = sum l_s 2^(m_s - M), o = sum o_s 2^(m_s - M)
  float4 hd[kMaxSplits];
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q)
    if (q < n_split)
      hd[q] = __ldcg(reinterpret_cast<const float4*>(a.attn_state) + ((slot * a.attn_splits + q) * (kWarps * 32) + tid) * 5);
  float MA = -INFINITY, MB = -INFINITY;
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q)
    if (q < n_split) {
      MA = fmaxf(MA, hd[q].x);
      MB = fmaxf(MB, hd[q].y);
    }
  lA = lB = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[j][i] = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q) {
    if (q >= n_split) break;
    const float wA = hd[q].x == -INFINITY ? 0.f : ex2(hd[q].x - MA);
    const float wB = hd[q].y == -INFINITY ? 0.f : ex2(hd[q].y - MB);
    lA += hd[q].z * wA;
    lB += hd[q].w * wB;
    const float4* so = reinterpret_cast<const float4*>(a.attn_state) + ((slot * a.attn_splits + q) * (kWarps * 32) + tid) * 5 + 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = __ldcg(so + j);
      o[j][0] += v.x * wA;
      o[j][1] += v.y * wA;
      o[j][2] += v.z * wB;
      o[j][3] += v.w * wB;
    }
  }
  if (tid == 0) a.attn_count[slot] = 0u;  // ready for the next call
  finish(r, Lr);
  publish();
}

}  // namespace

cudaError_t prepare_attention_kernel() {
  return cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_attention(const FwdArgs& a, __nv_bfloat16* zin, cudaStream_t s) {
  const int nblk = (a.B + kCandPerCta - 1) / kCandPerCta;
  return launch_kernel(attention_kernel, dim3(nblk, kG, a.attn_splits), dim3(kWarps * 32), kSmemBytes, s, a.pdl != 0,
                       a, zin);
}

}  // namespace cvr
