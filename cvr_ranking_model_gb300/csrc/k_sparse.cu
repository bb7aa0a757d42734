// Sparse side of the CVR forward pass and the small per-request GEMVs.
//
//  sparse_kernel       mean-pooled multi-hot embedding bags (user bags once per request, item bags per
//                      candidate; iQIYI ad-CVR article 3.1 item 2 and 3.4.5) with the [-clamp, clamp]
//                      clamp and bf16 cast after the lookup (GPU CTR inference article, section 三),
//                      plus the sequence-event gather from the shared id table (iQIYI 3.2.1): one launch
//                      for every lookup of the batch (iQIYI 3.4.2).
//  seq_colsum_kernel   partial column sums of the encoded sequences; the last block of each (request, group)
//                      forms the mean-pooled sequence vector and the mean-pool half of that group's query
//                      FFN, once per request (Query Decoding, iQIYI 3.2.3; the lazy user repeat of 3.4.5).
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kSparseThreads = 256;   // 8 warps
constexpr int kSparseBlocksPerSm = 3;  // persistent grid

__device__ __forceinline__ float clampf(float v, float c) { return fminf(fmaxf(v, -c), c); }

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float4 v) {
  uint2 p;
  p.x = pack_bf16(v.x, v.y);
  p.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = p;
}

// Persistent and software-pipelined: every warp walks units with a grid stride -- units of 4 bags (8 lanes
// per bag, each lane 4 of the 32 columns), then single sequence events -- and while the table rows of unit k
// are in flight it already loads the ids of unit k+1 and the offsets of unit k+2, so the three dependent
// round trips of a lookup (offsets -> ids -> rows) overlap instead of adding up.
__global__ void __launch_bounds__(kSparseThreads, kSparseBlocksPerSm) sparse_kernel(const __grid_constant__ FwdArgs a) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t gw = (int64_t)blockIdx.x * (kSparseThreads / 32) + (tid >> 5);
  const int64_t nw = (int64_t)gridDim.x * (kSparseThreads / 32);
  pdl_trigger();
  pdl_wait();
  // request ids: in range and non-decreasing (checked once per candidate)
  for (int64_t cand = (int64_t)blockIdx.x * kSparseThreads + tid; cand < a.B;
       cand += (int64_t)gridDim.x * kSparseThreads) {
    const int r = a.req_ids[cand];
    bool bad = r < 0 || r >= a.R;
    if (cand + 1 < a.B && a.req_ids[cand + 1] < r) bad = true;
    if (bad) atomicOr(a.err, kErrReqIds);
  }
  int errbits = 0;

  // ---------------------------------------------------------------- embedding bags
  {
    const int64_t n_user_bags = (int64_t)a.R * kFu;
    const int64_t n_bags = n_user_bags + (int64_t)a.B * kFi;
    const int64_t n_units = (n_bags + 3) / 4;
    const int grp = lane >> 3, sub = lane & 7;  // bag of this lane within the unit, its 4 columns
    auto bag_of = [&](int64_t u) { return min(u * 4 + grp, n_bags - 1); };
    int64_t u0 = gw, s0 = 0, e0 = 0, id0 = 0, s1 = 0, e1 = 0;
    if (u0 < n_units) {
      const int64_t b = bag_of(u0);
      s0 = a.bag_offsets[b];
      e0 = a.bag_offsets[b + 1];
    }
    if (u0 + nw < n_units) {
      const int64_t b = bag_of(u0 + nw);
      s1 = a.bag_offsets[b];
      e1 = a.bag_offsets[b + 1];
    }
    if (u0 < n_units && s0 + sub < e0) id0 = a.bag_ids[s0 + sub];
    while (u0 < n_units) {  // warp-uniform
      const int64_t u1 = u0 + nw, u2 = u1 + nw;
      // stage A: offsets of unit k+2; stage B: first ids of unit k+1 (raw; checked when used)
      int64_t s2 = 0, e2 = 0, id1 = 0;
      if (u2 < n_units) {
        const int64_t b = bag_of(u2);
        s2 = a.bag_offsets[b];
        e2 = a.bag_offsets[b + 1];
      }
      if (u1 < n_units && s1 + sub < e1) id1 = a.bag_ids[s1 + sub];
      // stage C: the rows of unit k
      const int64_t bag_raw = u0 * 4 + grp;
      const bool live = bag_raw < n_bags;  // dead lanes still take part in the shuffles
      const int64_t bag = live ? bag_raw : n_bags - 1;
      int field;
      __nv_bfloat16* dst;
      if (bag < n_user_bags) {
        field = (int)(bag % kFu);
        dst = a.U + (bag / kFu) * kUD + field * kE;
      } else {
        const int64_t ib = bag - n_user_bags;
        const int f = (int)(ib % kFi);
        field = kFu + f;
        dst = a.I + (ib / kFi) * kID + f * kE;
      }
      const float* table = a.tables[field];
      const int64_t rows = a.table_rows[field];
      const int64_t s = s0;
      int64_t e = e0;
      if (e < s) {
        if (live) errbits |= kErrOffsets;
        e = s;
      }
      // The 8 lanes of a bag hold 8 ids at once (one each), share them by shuffle, then have all 8 rows in
      // flight; the fp32 sum still runs in bag order from 0 (bit-exact with the definition). The loop count
      // is the warp's largest bag, so every lane reaches every shuffle.
      int64_t nmax = e - s;
      nmax = max(nmax, (int64_t)__shfl_xor_sync(0xffffffffu, (long long)nmax, 8));
      nmax = max(nmax, (int64_t)__shfl_xor_sync(0xffffffffu, (long long)nmax, 16));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int64_t base = 0; base < nmax; base += 8) {
        const int64_t j = s + base + sub;
        int64_t mine = 0;
        if (j < e) {
          mine = base == 0 ? id0 : a.bag_ids[j];
          if (mine < 0 || mine >= rows) {
            if (live) errbits |= kErrIdRange;
            mine = 0;
          }
          if (a.dbg_rows && live) a.dbg_rows[j] = mine;
        }
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int64_t id = __shfl_sync(0xffffffffu, (long long)mine, u, 8);
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (s + base + u < e) v[u] = __ldg(reinterpret_cast<const float4*>(table + id * kE) + sub);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (s + base + u < e) {
            acc.x = __fadd_rn(acc.x, v[u].x);
            acc.y = __fadd_rn(acc.y, v[u].y);
            acc.z = __fadd_rn(acc.z, v[u].z);
            acc.w = __fadd_rn(acc.w, v[u].w);
          }
        }
      }
      const int64_t n = e - s;
      float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n > 0) {
        const float fn = (float)n;
        m.x = __fdiv_rn(acc.x, fn);
        m.y = __fdiv_rn(acc.y, fn);
        m.z = __fdiv_rn(acc.z, fn);
        m.w = __fdiv_rn(acc.w, fn);
      }
      m.x = clampf(m.x, a.clamp);
      m.y = clampf(m.y, a.clamp);
      m.z = clampf(m.z, a.clamp);
      m.w = clampf(m.w, a.clamp);
      if (live) {
        store_bf16x4(dst + sub * 4, m);
        if (a.dbg_pooled) reinterpret_cast<float4*>(a.dbg_pooled + bag * kE)[sub] = m;
      }
      u0 = u1;
      s0 = s1;
      e0 = e1;
      id0 = id1;
      s1 = s2;
      e1 = e2;
    }
  }

  // ---------------------------------------------------------------- sequence events
  // one warp per event: 4 id columns -> 4 rows of the shared table -> one 128-wide row; the ids of the next
  // event load while this event's rows are in flight
  {
    const int64_t n_events = (int64_t)a.R * a.SL;
    const int c = lane >> 3, part = lane & 7;
    int64_t ev = gw;
    int64_t id_next = ev < n_events ? a.seq_ids[ev * kCols + c] : 0;
    while (ev < n_events) {  // warp-uniform
      const int64_t ev1 = ev + nw;
      int64_t id = id_next;
      id_next = ev1 < n_events ? a.seq_ids[ev1 * kCols + c] : 0;
      const int64_t r = ev / a.SL;
      int l = (int)(ev - r * a.SL);
      int g = 0;
      while (g < kG - 1 && l >= a.L[g]) {
        l -= a.L[g];
        ++g;
      }
      const int64_t row = a.goff[g] + r * a.L[g] + l;
      __nv_bfloat16* out = a.Xs + row * kD + c * kE + part * 4;
      bool pad = false;
      if (a.seq_lens) {
        const int raw = a.seq_lens[r * kG + g];
        if (l == 0 && lane == 0 && (raw < 0 || raw > a.L[g])) errbits |= kErrSeqLens;
        pad = l >= seq_len_of(a, r, g);  // padding: its id is never looked up; encoded from zeros, never used
      }
      if (pad) {
        store_bf16x4(out, make_float4(0.f, 0.f, 0.f, 0.f));
      } else {
        if (id < 0 || id >= a.table_rows[kFu + kFi]) {
          errbits |= kErrIdRange;
          id = 0;
        }
        float4 v = __ldg(reinterpret_cast<const float4*>(a.tables[kFu + kFi] + id * kE) + part);
        v.x = clampf(v.x, a.clamp);
        v.y = clampf(v.y, a.clamp);
        v.z = clampf(v.z, a.clamp);
        v.w = clampf(v.w, a.clamp);
        store_bf16x4(out, v);
      }
      ev = ev1;
    }
  }
  if (errbits) atomicOr(a.err, errbits);
}

// Partial column sums of H over chunks of 64 positions; grid (max_chunks, G, R), 128 threads. The last
// block of each (request, group) to finish -- found with a counter, nobody waits -- adds the partials up into
// the mean-pooled sequence vector m_g (iQIYI 3.2.3, Query Decoding item 1: mean over positions of the encoded
// states) and computes that group's per-request query term for every layer,
// qb[l][r][g*128 + n] = q_b[l][g*128 + n] + sum_k Wq[l][g][n][1664 + k] * m_g[k], then resets the counter.
__global__ void __launch_bounds__(128) seq_colsum_kernel(const __grid_constant__ FwdArgs a) {
  const int chunk = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const int L = a.L[g];
  const int t = threadIdx.x, cp = t & 63, half = t >> 6;
  // constants of the query term, loaded before waiting for the encoder (only the last block uses them):
  // row t of the first layer's mean-pool weights and its bias
  uint4 w0[16];
  {
    const uint4* wrow = reinterpret_cast<const uint4*>(a.qm + ((int64_t)g * kD + t) * kD);
#pragma unroll
    for (int v = 0; v < 16; ++v) w0[v] = __ldg(wrow + v);
  }
  const float qb0 = __ldg(a.q_b + g * kD + t);
  pdl_trigger();
  pdl_wait();
  // positions that count: the request's real events (all L without variable lengths); an empty group still
  // has one block, which writes a zero mean
  const int len = seq_len_of(a, r, g);
  const int chunks = len > 0 ? (len + 63) / 64 : 1;
  if (chunk >= chunks) return;
  const __nv_bfloat16* base = a.H + (a.goff[g] + (int64_t)r * L) * kD;
  const int l_end = min(len, chunk * 64 + 64);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
  for (int l = chunk * 64 + half; l < l_end; l += 2) {
    const __nv_bfloat162 v = __ldg(reinterpret_cast<const __nv_bfloat162*>(base + (int64_t)l * kD) + cp);
    s0 += __low2float(v);
    s1 += __high2float(v);
  }
  __shared__ float part[2][128];
  __shared__ float m[128];
  __shared__ int last;
  part[half][2 * cp] = s0;
  part[half][2 * cp + 1] = s1;
  __syncthreads();
  float* rg = a.colsum + ((int64_t)r * kG + g) * a.max_chunks * kD;
  rg[chunk * kD + t] = part[0][t] + part[1][t];
  __threadfence();
  __syncthreads();
  unsigned* cnt = a.cs_count + r * kG + g;
  if (t == 0) last = atomicAdd(cnt, 1u) == (unsigned)(chunks - 1);
  __syncthreads();
  if (!last) return;
  float sum = 0.f;
  for (int c0 = 0; c0 < chunks; c0 += 4) {  // four loads in flight, summed in chunk order
    float v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = c0 + c < chunks ? __ldcg(rg + (c0 + c) * kD + t) : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c0 + c < chunks) sum += v[c];
  }
  m[t] = len > 0 ? sum / (float)len : 0.f;
  if (t == 0) *cnt = 0u;
  __syncthreads();
  for (int l = 0; l < a.n_layers; ++l) {
    uint4 wv[16];
    if (l == 0) {
#pragma unroll
      for (int v = 0; v < 16; ++v) wv[v] = w0[v];
    } else {
      const uint4* wrow = reinterpret_cast<const uint4*>(a.qm + (((int64_t)l * kG + g) * kD + t) * kD);
#pragma unroll
      for (int v = 0; v < 16; ++v) wv[v] = __ldg(wrow + v);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&wv[v]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[q] += __low2float(e[q]) * m[v * 8 + 2 * q];
        acc[q] += __high2float(e[q]) * m[v * 8 + 2 * q + 1];
      }
    }
    a.qb[((int64_t)l * a.R + r) * (kG * kD) + g * kD + t] =
        (l == 0 ? qb0 : a.q_b[l * kG * kD + g * kD + t]) + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
  }
}

}  // namespace

cudaError_t launch_sparse(const FwdArgs& a, cudaStream_t s) {
  return launch_kernel(sparse_kernel, dim3(a.num_sms * kSparseBlocksPerSm), dim3(kSparseThreads), 0, s, false, a);
}

cudaError_t launch_seq_colsum(const FwdArgs& a, cudaStream_t s) {
  return launch_kernel(seq_colsum_kernel, dim3(a.max_chunks, kG, a.R), dim3(128), 0, s, a.pdl != 0, a);
}


}  // namespace cvr
