// Sparse side of the CVR forward pass and the small per-request GEMVs.
//
//  sparse_kernel       mean-pooled multi-hot embedding bags (user bags once per request, item bags per
//                      candidate; iQIYI ad-CVR article 3.1 item 2 and 3.4.5) with the [-clamp, clamp]
//                      clamp and bf16 cast after the lookup (GPU CTR inference article, section 三),
//                      plus the sequence-event gather from the shared id table (iQIYI 3.2.1): one launch
//                      for every lookup of the batch (iQIYI 3.4.2).
//  cache admission     the hot-row cache in HBM in front of tables kept in host memory (GPU CTR inference
//                      article, section 二: hot rows in HBM as the first tier, misses served from host DRAM)
//  seq_colsum_kernel   partial column sums of the encoded sequences; the last block of each (request, group)
//                      forms the mean-pooled sequence vector and the mean-pool half of that group's query
//                      FFN, once per request (Query Decoding, iQIYI 3.2.3; the lazy user repeat of 3.4.5).
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kSparseThreads = 256;   // 8 warps
constexpr int kSparseBlocksPerSm = 3;  // persistent grid

__device__ __forceinline__ float clampf(float v, float c) { return fminf(fmaxf(v, -c), c); }

// The gather's landing slots for embedding rows: per warp 2 units x [4 bags][8 rows][8 x 16 bytes] (dynamic
// shared memory, 64 KB per block).
constexpr int kSparseSmem = kSparseThreads / 32 * 2 * 4 * 8 * 8 * 16;
__device__ __forceinline__ float4* sparse_slots() {
  extern __shared__ float4 sparse_smem[];
  return sparse_smem;
}
__device__ __forceinline__ void sparse_cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void sparse_cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void sparse_cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float4 v) {
  uint2 p;
  p.x = pack_bf16(v.x, v.y);
  p.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = p;
}

// ---- hot-row cache: direct-mapped, slot = Fibonacci hash of the id. The cache is read-only during a call;
// a hit stamps the slot with the call's epoch, a miss reads the table row itself (host memory over C2C, or
// HBM) and logs (table, id) for admission after the call. Cached rows are exact copies, so a hit and a miss
// give the same bits.
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ int64_t cache_slot(int64_t id, int shift) {
  return (int64_t)(((uint64_t)id * kGolden) >> shift);
}

// Where the row of `id` in table t is read from; `hit`/`miss` say whether the table has a cache and which.
__device__ __forceinline__ const float* row_src(const FwdArgs& a, int t, int64_t id, unsigned epoch, bool mark,
                                                bool& hit, bool& miss) {
  const float* row = a.tables[t] + id * kE;
  const int64_t* tags = a.cache_tags[t];
  if (!tags) return row;
  const int64_t slot = cache_slot(id, a.cache_shift[t]);
  if (__ldcg(tags + slot) == id) {
    hit = true;
    if (mark) a.cache_use[t][slot] = epoch;
    return a.cache_rows[t] + slot * kE;
  }
  miss = true;
  return row;
}

// Logs the lanes' misses with one atomic per warp (entries past the log's capacity are not admitted).
__device__ __forceinline__ void log_misses(const FwdArgs& a, bool miss, int t, int64_t id, int lane) {
  const unsigned mb = __ballot_sync(0xffffffffu, miss);
  if (!mb) return;
  const int leader = __ffs(mb) - 1;
  unsigned base = 0;
  if (lane == leader) base = atomicAdd(a.cache_ctl, (unsigned)__popc(mb));
  base = __shfl_sync(0xffffffffu, base, leader);
  const unsigned idx = base + __popc(mb & ((1u << lane) - 1u));
  if (miss && idx < (unsigned)a.miss_cap) a.miss_list[idx] = ((int64_t)t << 48) | id;
}

__device__ __forceinline__ float4 ld_row(const float* p, int part, bool coherent) {
  return coherent ? __ldcg(reinterpret_cast<const float4*>(p) + part) : __ldg(reinterpret_cast<const float4*>(p) + part);
}

// Persistent and software-pipelined: every warp walks units with a grid stride -- units of 4 bags (8 lanes
// per bag, each lane 4 of the 32 columns), then single sequence events -- and while the table rows of unit k
// are in flight it already loads the ids of unit k+1 and the offsets of unit k+2, so the three dependent
// round trips of a lookup (offsets -> ids -> rows) overlap instead of adding up.
// kCache: some table has a hot-row cache (a separate instantiation keeps the plain path's registers as they are)
template <bool kCache>
__global__ void __launch_bounds__(kSparseThreads, kSparseBlocksPerSm) sparse_kernel(const __grid_constant__ FwdArgs a) {
  CVR_TL_BEGIN(TL_SPARSE);
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t gw = (int64_t)blockIdx.x * (kSparseThreads / 32) + (tid >> 5);
  const int64_t nw = (int64_t)gridDim.x * (kSparseThreads / 32);
  // The later kernels' weights (one packed allocation, a few MB) go to L2 while this kernel -- bound by the
  // latency of its dependent loads, not by bandwidth -- does its lookups: each block prefetches one slice
  // (256-byte aligned starts, sizes a multiple of 16 bytes, all inside the allocation).
  if (tid == 0 && a.wblob) {
    const int64_t slice = ((a.wblob_bytes + gridDim.x - 1) / gridDim.x + 255) / 256 * 256;
    const int64_t b0 = (int64_t)blockIdx.x * slice;
    const int64_t n = min(slice, a.wblob_bytes - b0) / 16 * 16;
    if (n > 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.wblob + b0), "r"((unsigned)n) : "memory");
  }
  pdl_trigger();
  pdl_wait();
  if (tid == 0) CVR_TL_WAITED();
  // the per-row-block counters that start the PLE block by block begin every call at zero
  if (a.ple_ready) {
    const int nrb = (a.B + 127) / 128;
    for (int i = blockIdx.x * kSparseThreads + tid; i < nrb; i += gridDim.x * kSparseThreads) {
      a.ple_ready[i] = 0u;
    }
  }
  if (a.attn_ready)  // and those that start the Token Mixer's tiles
    for (int i = blockIdx.x * kSparseThreads + tid; i < (a.B + 31) / 32; i += gridDim.x * kSparseThreads)
      a.attn_ready[i] = 0u;
  if (a.xu_ready)  // and so do the tokeniser's user row-tile flags
    for (int i = blockIdx.x * kSparseThreads + tid; i < (a.R + 127) / 128 * (kTokN / 128); i += gridDim.x * kSparseThreads)
      a.xu_ready[i] = 0u;
  if (a.cs_count)  // and the mean pool's per-(request, group) counters (also zeroed by whoever completes one)
    for (int i = blockIdx.x * kSparseThreads + tid; i < a.R * kG; i += gridDim.x * kSparseThreads) a.cs_count[i] = 0u;
  // request ids: in range and non-decreasing (checked once per candidate), and copied to the workspace for
  // the later kernels (the caller's array may be host memory read over the C2C link)
  for (int64_t cand = (int64_t)blockIdx.x * kSparseThreads + tid; cand < a.B;
       cand += (int64_t)gridDim.x * kSparseThreads) {
    const int r = a.req_in[cand];
    bool bad = r < 0 || r >= a.R;
    if (cand + 1 < a.B && a.req_in[cand + 1] < r) bad = true;
    if (bad) atomicOr(a.err, kErrReqIds);
    a.req_copy[cand] = r;
  }
  int errbits = 0;
  // with a cache, rows are read through L2 only (the admission after the previous call rewrote slots)
  constexpr bool cached = kCache;
  const unsigned epoch = cached ? a.cache_ctl[1] : 0u;
  unsigned long long n_hit = 0, n_miss = 0;

  // ---------------------------------------------------------------- embedding bags
  {
    const int64_t n_user_bags = (int64_t)a.R * kFu;
    const int64_t n_bags = n_user_bags + (int64_t)a.B * kFi;
    const int64_t n_units = (n_bags + 3) / 4;
    const int grp = lane >> 3, sub = lane & 7;  // bag of this lane within the unit, its 4 columns
    auto bag_of = [&](int64_t u) { return min(u * 4 + grp, n_bags - 1); };
    // A bag's [s, e) from the offsets. They are loaded two units ahead and checked one unit ahead, where they
    // are first used (so that the check does not wait for the load): a negative start or an end before the start
    // is reported and the bag is read as empty, so no id is ever read outside bag_ids.
    auto load_bag = [&](int64_t b, int64_t& s, int64_t& e) {
      s = a.bag_offsets[b];
      e = a.bag_offsets[b + 1];
    };
    auto check_bag = [&](int64_t& s, int64_t& e) {
      if (s < 0 || e < s) {
        errbits |= kErrOffsets;
        s = e = 0;
      }
    };
    // Where a bag's rows go: field, table rows, output row, for the bag of this lane in unit u.
    auto bag_place = [&](int64_t u, int& field, __nv_bfloat16*& dst) {
      const int64_t bag = bag_of(u);
      if (bag < n_user_bags) {
        field = (int)(bag % kFu);
        dst = a.U + (bag / kFu) * kUD + field * kE;
      } else {
        const int64_t ib = bag - n_user_bags;
        const int f = (int)(ib % kFi);
        field = kFu + f;
        dst = a.I + (ib / kFi) * kID + f * kE;
      }
    };
    // The address this lane's row slot reads (its id j = s + base + sub, checked; cache slot or table row),
    // or null when the bag has no row there. Counts and logs the cache's hits and misses (warp-collective).
    auto row_addr = [&](int64_t u, int64_t j, int64_t e, int64_t id, bool& bad) -> const float* {
      const bool live = u * 4 + grp < n_bags;
      int field;
      __nv_bfloat16* dst;
      bag_place(u, field, dst);
      const float* src = nullptr;
      bool hit = false, miss = false;
      int64_t mine = 0;
      if (j < e) {
        mine = id;
        if (mine < 0 || mine >= a.table_rows[field]) {
          if (live) bad = true;
          mine = 0;
        }
        if (a.dbg_rows && live) a.dbg_rows[j] = mine;
        src = kCache ? row_src(a, field, mine, epoch, live, hit, miss) : a.tables[field] + mine * kE;
      }
      if (cached) {
        miss = miss && live;
        n_hit += hit && live;
        n_miss += miss;
        log_misses(a, miss, field, mine, lane);
      }
      return src;
    };
    // Rows [s, s + 8) of each bag of unit u into one of this warp's two landing slots: lane `sub` copies the
    // 16-byte part `sub` of each row (the 8 lanes of a bag exchange the row addresses), so every lane later
    // reads only what it copied itself. One cp.async group per unit.
    float4* my_slots = sparse_slots() + (tid >> 5) * (2 * 4 * 8 * 8);
    auto issue_rows = [&](int64_t u, int64_t s, int64_t e, int64_t id, int slot) {
      bool bad = false;
      const float* src = u < n_units ? row_addr(u, s + sub, e, id, bad) : nullptr;
      if (bad) errbits |= kErrIdRange;
      float4* dst = my_slots + slot * (4 * 8 * 8) + grp * 64 + sub;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float* p = reinterpret_cast<const float*>(__shfl_sync(0xffffffffu, (long long)src, r, 8));
        if (s + r < e) sparse_cp_async16(dst + r * 8, p + sub * 4);
      }
      sparse_cp_async_commit();
    };
    // Pipeline per warp, unit k of its grid-stride sequence: offsets of k+3 load (raw), k+2's are checked and
    // its first ids load, k+1's rows are copied into a landing slot, and k's rows (copied one unit earlier) are
    // summed -- so two units of rows are in flight at once, without holding them in registers.
    int64_t s0 = 0, e0 = 0, s1 = 0, e1 = 0, s2 = 0, e2 = 0, id1 = 0;
    int64_t u0 = gw;
    if (u0 < n_units) load_bag(bag_of(u0), s0, e0);
    if (u0 + nw < n_units) load_bag(bag_of(u0 + nw), s1, e1);
    if (u0 + 2 * nw < n_units) load_bag(bag_of(u0 + 2 * nw), s2, e2);
    check_bag(s0, e0);
    check_bag(s1, e1);
    {
      int64_t id0 = 0;
      if (u0 < n_units && s0 + sub < e0) id0 = a.bag_ids[s0 + sub];
      if (u0 + nw < n_units && s1 + sub < e1) id1 = a.bag_ids[s1 + sub];
      if (u0 < n_units) issue_rows(u0, s0, e0, id0, 0);
    }
    int slot = 0;
    while (u0 < n_units) {  // warp-uniform
      const int64_t u1 = u0 + nw, u2 = u1 + nw, u3 = u2 + nw;
      int64_t s3 = 0, e3 = 0, id2 = 0;
      if (u3 < n_units) load_bag(bag_of(u3), s3, e3);
      check_bag(s2, e2);
      if (u2 < n_units && s2 + sub < e2) id2 = a.bag_ids[s2 + sub];
      if (u1 < n_units) issue_rows(u1, s1, e1, id1, slot ^ 1);
      // the rows of unit k: every group but the one just committed has landed
      if (u1 < n_units) sparse_cp_async_wait<1>();
      else sparse_cp_async_wait<0>();
      const bool live = u0 * 4 + grp < n_bags;
      int field;
      __nv_bfloat16* dst;
      bag_place(u0, field, dst);
      const int64_t bag = bag_of(u0);
      const int64_t s = s0, e = e0;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4* land = my_slots + slot * (4 * 8 * 8) + grp * 64 + sub;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (s + r < e) {  // the fp32 sum runs in bag order from 0 (bit-exact with the definition)
          const float4 v = land[r * 8];
          acc.x = __fadd_rn(acc.x, v.x);
          acc.y = __fadd_rn(acc.y, v.y);
          acc.z = __fadd_rn(acc.z, v.z);
          acc.w = __fadd_rn(acc.w, v.w);
        }
      }
      // bags of more than 8 ids: the rest in rounds of 8 read directly (the loop count is the warp's largest
      // bag, so every lane reaches every shuffle)
      int64_t nmax = e - s;
      nmax = max(nmax, (int64_t)__shfl_xor_sync(0xffffffffu, (long long)nmax, 8));
      nmax = max(nmax, (int64_t)__shfl_xor_sync(0xffffffffu, (long long)nmax, 16));
      for (int64_t base = 8; base < nmax; base += 8) {
        const int64_t j = s + base + sub;
        bool bad = false;
        const float* src = row_addr(u0, j, e, j < e ? a.bag_ids[j] : 0, bad);
        if (bad) errbits |= kErrIdRange;
        float4 v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float* p = reinterpret_cast<const float*>(__shfl_sync(0xffffffffu, (long long)src, r, 8));
          v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (s + base + r < e) v[r] = ld_row(p, sub, cached);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (s + base + r < e) {
            acc.x = __fadd_rn(acc.x, v[r].x);
            acc.y = __fadd_rn(acc.y, v[r].y);
            acc.z = __fadd_rn(acc.z, v[r].z);
            acc.w = __fadd_rn(acc.w, v[r].w);
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
      __syncwarp();  // (the slot just read is the next unit's landing slot)
      u0 = u1;
      s0 = s1;
      e0 = e1;
      s1 = s2;
      e1 = e2;
      id1 = id2;
      s2 = s3;
      e2 = e3;
      slot ^= 1;
    }
  }

  // ---------------------------------------------------------------- sequence events
  // a warp takes four events per round: per event 4 id columns -> 4 rows of the shared table -> one 128-wide row,
  // 8 lanes per row; each lane has its four events' rows in flight at once, and the next round's ids load
  // meanwhile
  {
    constexpr int kEvU = 4;
    const int64_t n_events = (int64_t)a.R * a.SL;
    const int c = lane >> 3, part = lane & 7;
    const int64_t stride = nw * kEvU;
    // The warps that walked one bag unit fewer (gw >= n_units % nw) come first. When the events fit in one round
    // of theirs (four each), they take them all and the warps with the most units take none; otherwise the
    // events go round-robin over all warps, those warps first, four per round. Events of a round: ev + u * step,
    // then ev += rstep.
    const int64_t n_units = ((int64_t)a.R * kFu + (int64_t)a.B * kFi + 3) / 4;
    const int64_t extra = n_units % nw;
    const bool one_round = extra > 0 && n_events <= kEvU * (nw - extra);
    int64_t ev = gw >= extra ? gw - extra : (one_round ? n_events : gw + (nw - extra));
    const int step = (int)(one_round ? nw - extra : nw), rstep = (int)(one_round ? n_events : stride);
    int64_t id_next[kEvU];
#pragma unroll
    for (int u = 0; u < kEvU; ++u) {
      const int64_t e = ev + u * step;
      id_next[u] = e < n_events ? a.seq_ids[e * kCols + c] : 0;
    }
    while (ev < n_events) {  // warp-uniform
      int64_t id[kEvU];
#pragma unroll
      for (int u = 0; u < kEvU; ++u) {
        id[u] = id_next[u];
        const int64_t e1 = ev + rstep + u * step;
        id_next[u] = e1 < n_events ? a.seq_ids[e1 * kCols + c] : 0;
      }
      __nv_bfloat16* out[kEvU];
      const float* src[kEvU];
#pragma unroll
      for (int u = 0; u < kEvU; ++u) {
        const int64_t e = ev + u * step;
        out[u] = nullptr;
        src[u] = nullptr;  // null: padding (stored as zeros) or past the last event
        bool hit = false, miss = false;
        if (e < n_events) {  // warp-uniform
          const int64_t r = e / a.SL;
          int l = (int)(e - r * a.SL);
          int g = 0;
          while (g < kG - 1 && l >= a.L[g]) {
            l -= a.L[g];
            ++g;
          }
          const int64_t row = a.goff[g] + r * a.L[g] + l;
          out[u] = a.Xs + row * kD + c * kE + part * 4;
          bool pad = false;
          if (a.seq_lens) {
            const int raw = a.seq_lens[r * kG + g];
            if (l == 0 && lane == 0 && (raw < 0 || raw > a.L[g])) errbits |= kErrSeqLens;
            pad = l >= seq_len_of(a, r, g);  // padding: its id is never looked up; encoded from zeros, never used
          }
          if (!pad) {
            int64_t iv = id[u];
            if (iv < 0 || iv >= a.table_rows[kFu + kFi]) {
              errbits |= kErrIdRange;
              iv = 0;
            }
            id[u] = iv;
            src[u] = kCache ? row_src(a, kFu + kFi, iv, epoch, part == 0, hit, miss) : a.tables[kFu + kFi] + iv * kE;
          }
        }
        if (cached) {  // one lane of each id's 8 counts and logs
          miss = miss && part == 0;
          n_hit += hit && part == 0;
          n_miss += miss;
          log_misses(a, miss, kFu + kFi, id[u], lane);
        }
      }
      float4 v[kEvU];
#pragma unroll
      for (int u = 0; u < kEvU; ++u) v[u] = src[u] ? ld_row(src[u], part, cached) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kEvU; ++u) {
        if (!out[u]) continue;
        v[u].x = clampf(v[u].x, a.clamp);
        v[u].y = clampf(v[u].y, a.clamp);
        v[u].z = clampf(v[u].z, a.clamp);
        v[u].w = clampf(v[u].w, a.clamp);
        store_bf16x4(out[u], v[u]);
      }
      ev += rstep;
    }
  }
  if (errbits) atomicOr(a.err, errbits);
  if (cached) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_hit += __shfl_xor_sync(0xffffffffu, n_hit, o);
      n_miss += __shfl_xor_sync(0xffffffffu, n_miss, o);
    }
    if (lane == 0 && (n_hit | n_miss)) {
      atomicAdd(a.cache_stat, n_hit);
      atomicAdd(a.cache_stat + 1, n_miss);
    }
  }
}

struct Claims {
  unsigned* p[kNTab];
};

// Admission, step 1: every logged miss whose slot was not read this call bids for it; the highest log index
// wins, so that exactly one row lands in each contested slot.
__global__ void __launch_bounds__(256) cache_claim_kernel(const __grid_constant__ FwdArgs a, Claims c) {
  pdl_trigger();
  pdl_wait();
  const unsigned n = min(a.cache_ctl[0], (unsigned)a.miss_cap), epoch = a.cache_ctl[1];
  for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int64_t e = a.miss_list[i];
    const int t = (int)(e >> 48);
    const int64_t id = e & ((int64_t(1) << 48) - 1);
    const int64_t slot = cache_slot(id, a.cache_shift[t]);
    if (a.cache_use[t][slot] != epoch) atomicMax(c.p[t] + slot, i + 1);
  }
}

// Admission, step 2: one warp per logged miss; the winner of a slot copies the row (32 floats) from the
// table and then sets the tag. The last block resets the log and moves to the next epoch.
__global__ void __launch_bounds__(256) cache_fill_kernel(const __grid_constant__ FwdArgs a, Claims c) {
  pdl_trigger();
  pdl_wait();
  const unsigned n = min(a.cache_ctl[0], (unsigned)a.miss_cap);
  const int lane = threadIdx.x & 31;
  const unsigned warps = gridDim.x * (blockDim.x / 32);
  for (unsigned i = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); i < n; i += warps) {
    const int64_t e = a.miss_list[i];
    const int t = (int)(e >> 48);
    const int64_t id = e & ((int64_t(1) << 48) - 1);
    const int64_t slot = cache_slot(id, a.cache_shift[t]);
    if (__ldcg(c.p[t] + slot) != i + 1) continue;  // warp-uniform
    const float v = a.tables[t][id * kE + lane];
    const_cast<float*>(a.cache_rows[t])[slot * kE + lane] = v;
    __syncwarp();
    if (lane == 0) {
      const_cast<int64_t*>(a.cache_tags[t])[slot] = id;
      c.p[t][slot] = 0u;
    }
  }
  cta_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.cache_ctl + 2, 1u) == gridDim.x - 1) {  // every block has read the log's length
      a.cache_ctl[0] = 0u;
      a.cache_ctl[1] += 1u;
      a.cache_ctl[2] = 0u;
    }
  }
}

// Column sums of H over chunks of kCsRows positions; grid (chunks, G, R), 512 threads. A (request, group) that
// fits one chunk (every one at the usual lengths) is summed by one block, which goes on directly; longer
// sequences write one partial sum per chunk and the last of their blocks -- found with a counter, nobody waits --
// adds the partials up in chunk order. That block then forms the mean-pooled sequence vector m_g (iQIYI 3.2.3,
// Query Decoding item 1: mean over positions of the encoded states) and that group's per-request query term
// for every layer, qb[l][r][g*128 + n] = q_b[l][g*128 + n] + sum_k Wq[l][g][n][1664 + k] * m_g[k].
constexpr int kCsRows = 512;
constexpr int kCsThreads = 512;

__global__ void __launch_bounds__(kCsThreads) seq_colsum_kernel(const __grid_constant__ FwdArgs a) {
  CVR_TL_BEGIN(TL_COLSUM);
  const int chunk = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const int L = a.L[g];
  const int t = threadIdx.x;
  // matvec thread t: output row n = t % 128, quarter t / 128 of K. The first layer's weights are constant: they
  // load while the encoder still runs
  const int nrow = t & (kD - 1), quarter = t >> 7;
  auto load_w = [&](uint4* wv, int l) {
    const uint4* wrow = reinterpret_cast<const uint4*>(a.qm + (((int64_t)l * kG + g) * kD + nrow) * kD + quarter * 32);
#pragma unroll
    for (int x = 0; x < 4; ++x) wv[x] = __ldg(wrow + x);
  };
  uint4 w0[4];
  load_w(w0, 0);
  pdl_trigger();
  pdl_wait();
  if (t == 0) CVR_TL_WAITED();
  // positions that count: the request's real events (all L without variable lengths); an empty group still
  // has one block, which writes a zero mean
  const int len = seq_len_of(a, r, g);
  const int chunks = len > 0 ? (len + kCsRows - 1) / kCsRows : 1;
  if (chunk >= chunks) return;
  const __nv_bfloat16* base = a.H + (a.goff[g] + (int64_t)r * L) * kD;
  const int l0 = chunk * kCsRows, l_end = min(len, l0 + kCsRows);
  // thread t sums columns [8 (t % 16), +8) over rows l0 + t/16 + 32 i, eight 16-byte loads in flight, in a fixed
  // order (the result does not depend on timing)
  const int cg = t & 15, rg = t >> 4;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int lb = l0 + rg; lb < l_end; lb += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int l = lb + 32 * i;
      v[i] = l < l_end ? __ldg(reinterpret_cast<const uint4*>(base + (int64_t)l * kD) + cg) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += __low2float(h[e]);
        acc[2 * e + 1] += __high2float(h[e]);
      }
    }
  }
  __shared__ float part[32][kD];
  __shared__ float m[kD];
  __shared__ float gpart[4][kD];
  __shared__ int last;
#pragma unroll
  for (int e = 0; e < 8; ++e) part[rg][cg * 8 + e] = acc[e];
  cta_sync();
  float colsum = 0.f;
  if (t < kD) {
#pragma unroll
    for (int j = 0; j < 32; ++j) colsum += part[j][t];
  }
  unsigned* cnt = a.cs_count + r * kG + g;
  if (chunks > 1) {
    float* rgp = a.colsum + ((int64_t)r * kG + g) * a.max_chunks * kD;
    if (t < kD) rgp[chunk * kD + t] = colsum;
    __threadfence();
    cta_sync();
    if (t == 0) last = atomicAdd(cnt, 1u) == (unsigned)(chunks - 1);
    cta_sync();
    if (!last) return;
    if (t < kD) {
      colsum = 0.f;
      for (int c = 0; c < chunks; ++c) colsum += __ldcg(rgp + c * kD + t);  // in chunk order
    }
    if (t == 0) *cnt = 0u;
  }
  if (t < kD) m[t] = len > 0 ? colsum / (float)len : 0.f;
  cta_sync();
  // the four quarters of K are added in a fixed order
  for (int l = 0; l < a.n_layers; ++l) {
    uint4 wv[4];
    if (l == 0) {
#pragma unroll
      for (int x = 0; x < 4; ++x) wv[x] = w0[x];
    } else {
      load_w(wv, l);
    }
    float s2[2] = {0.f, 0.f};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&wv[x]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = quarter * 32 + x * 8 + 2 * q;
        s2[q & 1] += __low2float(e[q]) * m[k];
        s2[q & 1] += __high2float(e[q]) * m[k + 1];
      }
    }
    gpart[quarter][nrow] = s2[0] + s2[1];
    cta_sync();
    if (t < kD)
      a.qb[((int64_t)l * a.R + r) * (kG * kD) + g * kD + t] =
          __ldg(a.q_b + l * kG * kD + g * kD + t) + ((gpart[0][t] + gpart[1][t]) + (gpart[2][t] + gpart[3][t]));
    cta_sync();
  }
}

}  // namespace

cudaError_t prepare_sparse_kernel() {
  cudaError_t e = cudaFuncSetAttribute(sparse_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSparseSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(sparse_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSparseSmem);
  // the column sums start on SMs the encoder has just left, which run with the largest shared-memory split: ask
  // for the same split, so that no SM has to change it first
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(seq_colsum_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t launch_sparse(const FwdArgs& a, cudaStream_t s) {
  return launch_kernel(a.cache_on ? sparse_kernel<true> : sparse_kernel<false>, dim3(a.num_sms * kSparseBlocksPerSm),
                       dim3(kSparseThreads), kSparseSmem, s, false, a);
}

cudaError_t launch_cache_admit(const FwdArgs& a, unsigned* const* claims, cudaStream_t s) {
  Claims c;
  for (int t = 0; t < kNTab; ++t) c.p[t] = claims[t];
  const dim3 grid(a.num_sms * 2), block(256);
  cudaError_t e = launch_kernel(cache_claim_kernel, grid, block, 0, s, a.pdl != 0, a, c);
  if (e == cudaSuccess) e = launch_kernel(cache_fill_kernel, grid, block, 0, s, a.pdl != 0, a, c);
  return e;
}

cudaError_t launch_seq_colsum(const FwdArgs& a, cudaStream_t s) {
  return launch_kernel(seq_colsum_kernel, dim3(a.max_chunks, kG, a.R), dim3(kCsThreads), 0, s, a.pdl != 0, a);
}


}  // namespace cvr
