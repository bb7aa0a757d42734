// Query Decoding cross-attention on tcgen05 (iQIYI ad-CVR article, section 3.2.3): for every candidate and
// group g, the group's query (4 heads of 32) attends over that request's encoded sequence H_g, which serves
// as both K and V; logits are scaled by 1/(tau*sqrt(32)) and normalised by a softmax over the sequence.
//
// One CTA = one group x 128 consecutive candidates (the M of the MMAs) x one request. Per chunk of 64 positions:
//   S_h = Q_h K_h^T      4 heads x (M=128, N=64, K=32) into TMEM columns [64h, 64h+64)
//   softmax             8 warps in two groups, group p owning heads 2p and 2p+1; a thread holds one candidate
//                       row and reads S straight from TMEM, so the row max and sum need no shuffles;
//                       P_h = exp2(S_h - m_h) in bf16 into shared memory (the A operand of P.V)
//   O_h += P_h V_h      4 heads x (M=128, N=32, K=64) into TMEM columns [256 + 32h, ...), V_h^T read from a
//                       K-major copy that 2 more warps transpose from the chunk
// Warp 0 streams Q (once) and the K/V chunks by TMA into a double buffer; warp 1 issues the MMAs head by
// head, P_h V_h of the previous chunk just before S_h of the next, so that one commit after S_h tells the
// softmax warps both that S_h is ready and that P_h may be overwritten and O_h is up to date. A softmax
// group alternates between its two heads, which hides the MMA round trip of one behind the other. With head
// dimension 32 a position costs 128 flops on the tensor cores against one exponential, so the softmax warps
// set the pace: the scale is folded into one FMA per logit and the max is taken on the raw logits (the
// scale is positive). The running max m_h of
// a row only moves when a chunk's max exceeds it by more than 8 (in log2 units): P stays below 2^8 and O
// needs rescaling only then (O and l use the same m_h, so the result is exact up to rounding). A tile
// holding candidates of several requests is processed once per request (rows of other requests are not
// stored); a group longer than 512 positions is split over several CTAs whose states the last one merges.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kRows = 128;                 // candidates per CTA
constexpr int kKeys = 64;                  // positions per chunk
constexpr int kPairs = 2;                  // softmax groups, two heads each
constexpr int kThreads = 384;              // warp 0 TMA, 1 MMA, 2..3 V transpose, 4..11 softmax (3 warps per SMSP)
constexpr int kSoftWarp0 = 4;
constexpr int kTrWarps = 2;
constexpr int kQBytes = kRows * kD * 2;    // 32 KB: 2 swizzle atoms of [128 rows][64 dims]
constexpr int kKVBytes = kKeys * kD * 2;   // 16 KB: 2 atoms of [64 positions][64 dims]
constexpr int kVTBytes = kD * kKeys * 2;   // 16 KB: [128 dims][64 positions]
constexpr int kPBytes = kRows * kKeys * 2;  // 16 KB per head: [128 rows][64 positions]
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffVT = kOffKV + 2 * kKVBytes;
constexpr int kOffP = kOffVT + 2 * kVTBytes;
constexpr int kOffBar = kOffP + kHeads * kPBytes;
constexpr int kNBar = 24;
constexpr int kSmemBytes = 1024 + kOffBar + kNBar * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
static_assert(kKeys == kAttnChunk, "split sizing uses the same chunk");
static_assert(kAttnCounters == kPairs * 4, "one merge counter per softmax warp");
// TMEM: S 4 heads x 64 columns, O 4 x 32
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleLog2 = 8.f;        // a row max moves only when a chunk exceeds it by this much
constexpr int kStateF4 = kAttnStateFloats / 4;  // split state of a row: m[4], l[4], O[4][32]
// MMA issue order of the heads, 0 2 1 3: the two softmax groups' first heads come first
__device__ __forceinline__ int head_order(int i) { return ((i & 1) << 1) | (i >> 1); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The softmax of one head on one 64-position chunk: returns the row sum of P and writes P (bf16, swizzled) to
// prow. m is the running max in scaled log2 units; positions at or past `valid` get P = 0.
template <bool kTail>
__device__ __forceinline__ float softmax_chunk(const uint32_t (&v)[kKeys], float sl2, float m, int valid,
                                               uint8_t* prow, int rl) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  const float nm = -m;
#pragma unroll
  for (int j = 0; j < kKeys / 8; ++j) {
    float p[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = j * 8 + e;
      p[e] = ex2(fmaf(__uint_as_float(v[k]), sl2, nm));
      if (kTail) p[e] = k < valid ? p[e] : 0.f;
    }
    s0 += p[0] + p[4];
    s1 += p[1] + p[5];
    s2 += p[2] + p[6];
    s3 += p[3] + p[7];
    *reinterpret_cast<uint4*>(prow + ((j ^ (rl & 7)) << 4)) =
        make_uint4(pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]), pack_bf16(p[4], p[5]), pack_bf16(p[6], p[7]));
  }
  return (s0 + s1) + (s2 + s3);
}

template <bool kTail>
__device__ __forceinline__ float raw_max(const uint32_t (&v)[kKeys], int valid) {
  float x0 = -INFINITY, x1 = -INFINITY, x2 = -INFINITY, x3 = -INFINITY;
#pragma unroll
  for (int k = 0; k < kKeys; k += 4) {
    float a0 = __uint_as_float(v[k]), a1 = __uint_as_float(v[k + 1]);
    float a2 = __uint_as_float(v[k + 2]), a3 = __uint_as_float(v[k + 3]);
    if (kTail) {
      a0 = k < valid ? a0 : -INFINITY;
      a1 = k + 1 < valid ? a1 : -INFINITY;
      a2 = k + 2 < valid ? a2 : -INFINITY;
      a3 = k + 3 < valid ? a3 : -INFINITY;
    }
    x0 = fmaxf(x0, a0);
    x1 = fmaxf(x1, a1);
    x2 = fmaxf(x2, a2);
    x3 = fmaxf(x3, a3);
  }
  return fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
}

__device__ __forceinline__ void store_head_row(uint4* dst, const float (&o)[kHD], float inv) {
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint4 pq;
    pq.x = pack_bf16(o[8 * x] * inv, o[8 * x + 1] * inv);
    pq.y = pack_bf16(o[8 * x + 2] * inv, o[8 * x + 3] * inv);
    pq.z = pack_bf16(o[8 * x + 4] * inv, o[8 * x + 5] * inv);
    pq.w = pack_bf16(o[8 * x + 6] * inv, o[8 * x + 7] * inv);
    dst[x] = pq;
  }
}

__global__ void __launch_bounds__(kThreads, 1) attention_tc_kernel(const __grid_constant__ FwdArgs a,
                                                                   const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmH,
                                                                   __nv_bfloat16* __restrict__ zin) {
  extern __shared__ uint8_t smem_raw[];
  CVR_TL_BEGIN(TL_ATTENTION_TC);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKV = smem + kOffKV;
  uint8_t* sVT = smem + kOffVT;
  uint8_t* sP = smem + kOffP;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bar;          // Q landed
  uint64_t* kv_full = bar + 1;     // [2] chunk landed
  uint64_t* kv_empty = bar + 3;    // [2] S MMAs and the transpose are done with it
  uint64_t* vt_full = bar + 5;     // [2] V^T written
  uint64_t* vt_empty = bar + 7;    // [2] the P.V MMAs that read V^T have completed
  uint64_t* s_full = bar + 9;      // [head] S_h ready; every earlier MMA (P_h V_h of the chunk before) done
  uint64_t* p_full = bar + 13;     // [head] P_h written to shared memory (S_h has been read)
  uint64_t* o_full = bar + 17;     // the last P.V MMAs of a request's pass completed
  uint64_t* o_empty = bar + 18;    // softmax has read O (a next request's pass may overwrite it)
  uint64_t* drained = bar + 19;    // after an abort: every MMA issued so far has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int g = a.g_order[blockIdx.y], sp = blockIdx.z;
  const int b0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = a.L[g];
  const int n_split = split_count(L);
  pdl_trigger();
  if (sp >= n_split) return;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1 + kTrWarps);
      mbar_init(&vt_full[i], kTrWarps);
      mbar_init(&vt_empty[i], 1);
    }
    for (int h = 0; h < kHeads; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, 8);
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmH);
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  pdl_wait();
  if (threadIdx.x == 0) CVR_TL_WAITED();

  const int B = a.B, R = a.R;
  const int b_last = min(b0 + kRows, B) - 1;
  // request ids are validated by the sparse kernel; here they are only kept in range
  const int r_first = min(max(a.req_ids[b0], 0), R - 1);
  const int r_last = min(max(a.req_ids[b_last], 0), R - 1);
  const bool split = n_split > 1 && r_first == r_last;
  const bool skip = !split && sp > 0;  // (the first split's CTA takes every position of a multi-request tile)
  const int per = ((L + kKeys - 1) / kKeys + n_split - 1) / n_split;  // chunks per split

  // chunk range of request r for this CTA
  auto range = [&](int r, int& c0, int& c1, int& Lr) {
    Lr = seq_len_of(a, r, g);
    const int nch = (Lr + kKeys - 1) / kKeys;
    c0 = split ? min(sp * per, nch) : 0;
    c1 = split ? min((sp + 1) * per, nch) : nch;
  };

  int n_loaded = 0;  // chunks the TMA warp issued
  if (!skip && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(q_full, kQBytes);
      for (int at = 0; at < 2; ++at) tma_load_2d(sQ + at * (kRows * 128), &tmQ, q_full, g * kD + at * 64, b0);
    }
    int t = 0;  // chunks streamed so far (buffer t % 2)
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      int c0, c1, Lr;
      range(r, c0, c1, Lr);
      const int row0 = (int)(a.goff[g] + (int64_t)r * L);
      for (int c = c0; c < c1; ++c, ++t) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait_warp(&kv_empty[s], ((t >> 1) - 1) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(&kv_full[s], kKVBytes);
          for (int at = 0; at < 2; ++at)
            tma_load_2d(sKV + s * kKVBytes + at * (kKeys * 128), &tmH, &kv_full[s], at * 64, row0 + c * kKeys);
        }
        __syncwarp();
      }
    }
    n_loaded = t;
  } else if (!skip && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = idesc_bf16(kRows, kKeys), id_o = idesc_bf16(kRows, kHD);
    bool ok = mbar_wait_warp(q_full, 0, abort_flag, a.err);
    int t = 0, npass = 0;
    // O_h (+)= P_h V_h of chunk tp, once the softmax has written P_h
    auto issue_pv = [&](int tp, int h, bool first) -> bool {
      if (!mbar_wait_warp(&p_full[h], tp & 1, abort_flag, a.err)) return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          tc_mma(tbase + kColO + h * kHD, sdesc_sw128(smem_u32(sP + h * kPBytes) + k * 32),
                 sdesc_sw128(smem_u32(sVT + (tp & 1) * kVTBytes + h * kHD * 128) + k * 32), id_o,
                 (!first || k > 0) ? 1u : 0u);
      }
      __syncwarp();
      return true;
    };
    // the start of chunk tp's P.V MMAs: its V^T is written, and the previous pass's O has been read
    auto pv_ready = [&](int tp, bool& need_o_empty) -> bool {
      if (!mbar_wait_warp(&vt_full[tp & 1], (tp >> 1) & 1, abort_flag, a.err)) return false;
      if (need_o_empty && !mbar_wait_warp(o_empty, (npass - 2) & 1, abort_flag, a.err)) return false;
      need_o_empty = false;
      return true;
    };
    for (int r = r_first; r <= r_last && ok; ++r) {
      int c0, c1, Lr;
      range(r, c0, c1, Lr);
      if (c0 >= c1) continue;
      ++npass;
      bool need_o_empty = npass > 1;
      const int tfirst = t;
      for (int c = c0; c < c1 && ok; ++c, ++t) {
        const int s = t & 1;
        ok = mbar_wait_warp(&kv_full[s], (t >> 1) & 1, abort_flag, a.err);
        const bool pv = t > tfirst;  // P.V of the previous chunk goes in before each head's next S
        if (ok && pv) ok = pv_ready(t - 1, need_o_empty);
        for (int i = 0; i < kHeads && ok; ++i) {
          const int h = head_order(i);
          if (pv) ok = issue_pv(t - 1, h, t - 1 == tfirst);
          if (!ok) break;
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kHD / 16; ++k)
              tc_mma(tbase + kColS + h * kKeys,
                     sdesc_sw128(smem_u32(sQ + (h >> 1) * (kRows * 128)) + (h & 1) * 64 + k * 32),
                     sdesc_sw128(smem_u32(sKV + s * kKVBytes + (h >> 1) * (kKeys * 128)) + (h & 1) * 64 + k * 32),
                     id_s, k > 0 ? 1u : 0u);
            tc_commit(&s_full[h]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          if (pv) tc_commit(&vt_empty[(t - 1) & 1]);
          tc_commit(&kv_empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      // the pass's last chunk
      ok = pv_ready(t - 1, need_o_empty);
      for (int i = 0; i < kHeads && ok; ++i) ok = issue_pv(t - 1, head_order(i), t - 1 == tfirst);
      if (!ok) break;
      if (lane == 0) {
        tc_commit(&vt_empty[(t - 1) & 1]);
        tc_commit(o_full);
      }
      __syncwarp();
    }
  } else if (!skip && warp < kSoftWarp0) {
    // ------------------------------------------------------------ V transpose: thread = dims d and d + 64
    const int d = (warp - 2) * 32 + lane;
    const int cb = d >> 3, e = d & 7;
    int t = 0;
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      int c0, c1, Lr;
      range(r, c0, c1, Lr);
      for (int c = c0; c < c1; ++c, ++t) {
        const int s = t & 1;
        ok = mbar_wait_warp(&kv_full[s], (t >> 1) & 1, abort_flag, a.err);
        // V^T buffer s was last read by the P.V of chunk t - 2
        if (ok && t >= 2) ok = mbar_wait_warp(&vt_empty[s], ((t >> 1) - 1) & 1, abort_flag, a.err);
        if (!ok) break;
#pragma unroll
        for (int at = 0; at < 2; ++at) {
          const uint8_t* src = sKV + s * kKVBytes + at * (kKeys * 128);
          uint8_t* dst = sVT + s * kVTBytes + (d + 64 * at) * 128;
#pragma unroll
          for (int j = 0; j < kKeys / 8; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int k0 = j * 8 + 2 * q, k1 = k0 + 1;
              const uint16_t lo = *reinterpret_cast<const uint16_t*>(src + k0 * 128 + ((cb ^ (k0 & 7)) << 4) + e * 2);
              const uint16_t hi = *reinterpret_cast<const uint16_t*>(src + k1 * 128 + ((cb ^ (k1 & 7)) << 4) + e * 2);
              w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            // (d + 64 at) & 7 == d & 7
            *reinterpret_cast<uint4*>(dst + ((j ^ (d & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&vt_full[s]);
          mbar_arrive(&kv_empty[s]);
        }
      }
    }
  } else if (!skip) {
    // ------------------------------------------------------------ softmax + output: thread = candidate row
    const int sw = warp - kSoftWarp0, pair = sw >> 2;
    const int q = warp & 3, rl = q * 32 + lane, row = b0 + rl;  // TMEM lane quarter of this warp
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int req = row < B ? a.req_ids[row] : -1;
    // logits * log2(e) / (tau * sqrt(head_dim)) so that the softmax runs on exp2
    const float sl2 = 1.4426950408889634f / (a.tau * sqrtf((float)kHD));
    int t = 0, np = 0;
    bool ok = true;
    for (int r = r_first; r <= r_last && ok; ++r) {
      int c0, c1, Lr;
      range(r, c0, c1, Lr);
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // the pair's two heads
      const int tfirst = t;
      for (int c = c0; c < c1 && ok; ++c, ++t) {
        const int valid = Lr - c * kKeys;  // positions of this chunk inside the sequence (>= 1)
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 2 * pair + hh;
          // S_h of this chunk; its commit also covers P_h V_h of the previous chunk (P_h's buffer free, O_h current)
          ok = mbar_wait_warp(&s_full[h], t & 1, abort_flag, a.err);
          if (!ok) break;
          tc_fence_after();
          uint32_t v[kKeys];
          tmem_ld32_nowait(tbase + lane_off + kColS + h * kKeys, v);
          tmem_ld32_nowait(tbase + lane_off + kColS + h * kKeys + 32, v + 32);
          tmem_ld_wait();
          const float mx = (valid >= kKeys ? raw_max<false>(v, valid) : raw_max<true>(v, valid)) * sl2;
          float mh = hh ? m1 : m0;
          // TMEM loads and stores are warp-collective: when any row's max moves, the whole warp rescales, each
          // row to its own new max (a factor of 1 where the max stayed)
          if (__any_sync(0xffffffffu, mx > mh + kRescaleLog2)) {
            const float mn = fmaxf(mh, mx);
            if (t > tfirst) {
              const float f = ex2(mh - mn);
              uint32_t ov[32];
              tmem_ld32_nowait(tbase + lane_off + kColO + h * kHD, ov);
              tmem_ld_wait();
#pragma unroll
              for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * f);
              tmem_st16(tbase + lane_off + kColO + h * kHD, ov);
              tmem_st16(tbase + lane_off + kColO + h * kHD + 16, ov + 16);
              if (hh) l1 *= f;
              else l0 *= f;
            }
            mh = mn;
            if (hh) m1 = mn;
            else m0 = mn;
          }
          uint8_t* prow = sP + h * kPBytes + rl * 128;
          const float sum = valid >= kKeys ? softmax_chunk<false>(v, sl2, mh, valid, prow, rl)
                                           : softmax_chunk<true>(v, sl2, mh, valid, prow, rl);
          if (hh) l1 += sum;
          else l0 += sum;
          tmem_st_wait();  // (a rescale of O_h above)
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[h]);
        }
      }
      if (!ok) break;
      // ---- this request's result (or this split's state) for the pair's heads
      const bool any = c1 > c0;
      if (any) {
        ok = mbar_wait_warp(o_full, np & 1, abort_flag, a.err);
        if (!ok) break;
        ++np;
        tc_fence_after();
      }
      const int64_t slot = (int64_t)blockIdx.x * kG + g;
      float4* st = reinterpret_cast<float4*>(a.attn_state) + ((slot * a.attn_splits + sp) * kRows + rl) * kStateF4;
      uint4* dst = reinterpret_cast<uint4*>(zin + (int64_t)row * kYD + kXD + g * kD);
      const bool store_row = req == r && row < B;
      if (split) {
        reinterpret_cast<float2*>(st)[pair] = make_float2(m0, m1);
        reinterpret_cast<float2*>(st + 1)[pair] = make_float2(l0, l1);
      }
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * pair + hh;
        float o[kHD];
        if (any) {
          uint32_t ov[32];
          tmem_ld32_nowait(tbase + lane_off + kColO + h * kHD, ov);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < kHD; ++x) o[x] = __uint_as_float(ov[x]);
        } else {
#pragma unroll
          for (int x = 0; x < kHD; ++x) o[x] = 0.f;
        }
        if (split) {
#pragma unroll
          for (int x = 0; x < 8; ++x) st[2 + h * 8 + x] = make_float4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
        } else if (store_row) {
          // decoded token g: head h in columns [32h, 32h+32) of slot 13 + g; no event -> zero token
          const float lh = hh ? l1 : l0;
          store_head_row(dst + h * 4, o, Lr > 0 ? 1.f / lh : 0.f);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && any) mbar_arrive(o_empty);
      if (!split) continue;
      // Each softmax warp counts its own (rows, heads) over the splits: the warp that completes them merges in
      // split order, M = max m_s, l = sum l_s 2^(m_s - M), O = sum O_s 2^(m_s - M) (nobody waits).
      __threadfence();
      __syncwarp();
      unsigned* cnt = a.attn_count + slot * kAttnCounters + sw;
      int last = 0;
      if (lane == 0) last = atomicAdd(cnt, 1u) == (unsigned)(n_split - 1);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) break;
      __threadfence();
      const float4* sbase = reinterpret_cast<const float4*>(a.attn_state) + (slot * a.attn_splits * kRows + rl) * kStateF4;
      const int64_t sstride = (int64_t)kRows * kStateF4;  // float4s from one split's state to the next
      float2 mm[kMaxSplits], ll[kMaxSplits];
#pragma unroll
      for (int qs = 0; qs < kMaxSplits; ++qs) {
        mm[qs] = make_float2(-INFINITY, -INFINITY);
        ll[qs] = make_float2(0.f, 0.f);
        if (qs < n_split) {
          mm[qs] = __ldcg(reinterpret_cast<const float2*>(sbase + qs * sstride) + pair);
          ll[qs] = __ldcg(reinterpret_cast<const float2*>(sbase + qs * sstride + 1) + pair);
        }
      }
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * pair + hh;
        float M = -INFINITY;
#pragma unroll
        for (int qs = 0; qs < kMaxSplits; ++qs) M = fmaxf(M, hh ? mm[qs].y : mm[qs].x);
        float o[kHD], lh = 0.f;
#pragma unroll
        for (int x = 0; x < kHD; ++x) o[x] = 0.f;
#pragma unroll
        for (int qs = 0; qs < kMaxSplits; ++qs) {
          if (qs >= n_split) break;
          const float ms = hh ? mm[qs].y : mm[qs].x;
          const float w = ms == -INFINITY ? 0.f : ex2(ms - M);
          lh += (hh ? ll[qs].y : ll[qs].x) * w;
          const float4* sq = sbase + qs * sstride + 2 + h * 8;
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float4 ov = __ldcg(sq + x);
            o[4 * x] += ov.x * w;
            o[4 * x + 1] += ov.y * w;
            o[4 * x + 2] += ov.z * w;
            o[4 * x + 3] += ov.w * w;
          }
        }
        if (store_row) store_head_row(dst + h * 4, o, Lr > 0 ? 1.f / lh : 0.f);
      }
      if (lane == 0) *cnt = 0u;  // ready for the next call
    }
  }
  cta_sync();
  if (*abort_flag && !skip && lane == 0) {
    // a wait gave up: let this CTA's own loads and MMAs land before its shared memory and TMEM are released
    if (warp == 0) {
      mbar_drain(q_full, 0);
      for (int t = n_loaded > 2 ? n_loaded - 2 : 0; t < n_loaded; ++t) mbar_drain(&kv_full[t & 1], (t >> 1) & 1);
    } else if (warp == 1) {
      tc_commit(drained);
      mbar_drain(drained, 0);
    }
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

cudaError_t prepare_attention_tc_kernel() {
  return cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_attention_tc(const FwdArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmH,
                                __nv_bfloat16* zin, cudaStream_t s) {
  const int nblk = (a.B + kRows - 1) / kRows;
  return launch_kernel(attention_tc_kernel, dim3(nblk, kG, a.attn_splits), dim3(kThreads), kSmemBytes, s,
                       a.pdl != 0, a, tmQ, tmH, zin);
}

}  // namespace cvr
