// Fused SwiGLU 128 -> 256 -> 128 on tcgen05, used twice in the CVR forward pass:
//
//  SEQ  the per-group sequence encoder (iQIYI ad-CVR article 3.2.2: each behaviour sequence is mapped
//       position-wise into the token space by its own SwiGLU): rows = sequence events of one group,
//       output H = W2 (silu(W1 x + b1) * (W3 x + b3)) + b2.
//  TM   the Query Boosting Token Mixer (iQIYI 3.2.3): the A operand is Mix(Z) -- 16 tokens x 16 heads of
//       8 transposed. The epilogue warps, which load Z anyway for the residual, write it into tensor memory
//       in mixed order (token t, head j of candidate b becomes K-slot t of mixed row (b, j)); the epilogue
//       applies the inverse map (Revert), the residual and the RMSNorm and writes Y in the original order.
//
// Persistent and warp-specialised: one CTA per SM loops over 128-row tiles. All SwiGLU weights (W1/W3 128 KB,
// W2 64 KB) stay resident in shared memory (reloaded only when a sequence tile changes group). The hidden
// width is processed in 2 chunks of 128 units: the up projection of a chunk is one chain of N=256 MMAs
// (128 W1 rows + 128 W3 rows, K=128) into the TMEM up-buffer; sixteen epilogue warps turn it into
// silu(a)*g and store the bf16 hidden chunk back into TMEM, where it is the A operand of the down
// projection (8 MMAs, K=16 each) accumulating into the TMEM down-buffer. The MMA warp issues the next
// chunk's up projection as soon as the epilogue has read the up-buffer, then the current chunk's down
// projection, so the tensor pipe works while the epilogue computes. Few, wide MMAs and two handshakes per
// chunk keep the single issuing thread ahead of the tensor pipe.
// TMEM: up 256, down 128, hidden 64, mixed activations 64 columns.
#include "cvr_internal.cuh"

namespace cvr {

namespace {

constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + kEpiWarps * 32;   // warp 0: TMA, warp 1: MMA, warps 2..17: epilogue
constexpr int kChunks = 2;                      // hidden chunks of 128
constexpr int kATile = 128 * kD * 2;            // 32 KB
constexpr int kW13Bytes = 2 * kHid * kD * 2;    // 128 KB: chunk c, K-block kb = [W1 64 ; W3 64 ; W1 64 ; W3 64] x 64
constexpr int kW2Bytes = kD * kHid * 2;         // 64 KB: 4 K-blocks of [128][64]
constexpr int kOffA = 0;
constexpr int kOffW13 = kOffA + kATile;
constexpr int kOffW2 = kOffW13 + kW13Bytes;
constexpr int kOffBias = kOffW2 + kW2Bytes;     // fp32 b1/b3 [512] (interleaved like W13) + b2 [128] of one group
constexpr int kBiasFloats = 2 * kHid + kD;
constexpr int kOffBar = kOffBias + kBiasFloats * 4;
constexpr int kNBar = 10;
// The dynamic shared-memory window is 1024-byte aligned (checked at run time; the kernel reports an error
// and does nothing otherwise), so no alignment slack is requested: the whole 227 KB budget is used.
constexpr int kSmemBytes = kOffBar + kNBar * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
// TMEM column bases. SEQ: hidden chunk at 384. TM: mixed activations of even / odd tiles at 384 / 448 (the
// hidden chunk goes to shared memory instead).
constexpr uint32_t kColUp = 0, kColDown = 256, kColHid = 384, kColA = 384;

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
__device__ __forceinline__ void epi_sync() {
  __syncwarp();  // (the warp arrives converged)
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    swiglu_mlp_kernel(const __grid_constant__ FwdArgs a, const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2, int layer,
                      int n_tiles, int n_cta, const __nv_bfloat16* __restrict__ zin, __nv_bfloat16* __restrict__ yout) {
  extern __shared__ __align__(1024) uint8_t smem[];
  CVR_TL_BEGIN(MODE == MODE_SEQ ? TL_SEQ_MLP : TL_TOKEN_MIXER);
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
  uint64_t* a_full = bar;              // activation tile landed (SEQ: TMA; TM: epilogue warps)
  uint64_t* a_empty = bar + 1;         // last up MMA of the tile has read it
  uint64_t* w_full = bar + 2;          // weights landed
  uint64_t* w_empty = bar + 3;         // weights may be replaced (sequence group change)
  uint64_t* up_full = bar + 4;         // up accumulator ready
  uint64_t* up_empty = bar + 5;        // epilogue has read it
  uint64_t* hm_full = bar + 6;         // hidden chunk stored in TMEM
  uint64_t* hm_empty = bar + 7;        // down MMAs have read it
  uint64_t* dn_full = bar + 8;         // down accumulator ready
  uint64_t* dn_empty = bar + 9;        // epilogue has read it
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  unsigned* ydone = tslot + 2;  // TM: epilogue-warp parts of tiles written (16 per tile)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(a_full, MODE == MODE_TM ? kEpiWarps : 1);
    mbar_init(a_empty, 1);
    mbar_init(w_full, 1);
    mbar_init(w_empty, 1);
    mbar_init(up_full, 1);
    mbar_init(up_empty, kEpiWarps);
    mbar_init(hm_full, kEpiWarps);
    mbar_init(hm_empty, 1);
    mbar_init(dn_full, 1);
    mbar_init(dn_empty, kEpiWarps);
    *abort_flag = 0;
    *ydone = 0u;
    fence_mbar_init();
    if (MODE == MODE_SEQ) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW13);
    tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  // The Token Mixer lets the next kernel (the PLE, which starts row block by row block) launch at once. The sequence
  // encoder lets its dependents launch only when its epilogue has finished its tiles: their CTAs then take the SMs
  // this kernel leaves, instead of SMs that a kernel on another stream is about to need.
  if (MODE == MODE_TM) pdl_trigger();
  const int n_my = (int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / n_cta + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (it stays converged); lane 0 issues the copies. Weights are constant, so
    // their loads may start before the previous kernel has finished; activation loads wait for it first.
    int w_group = -1, w_loads = 0;
    bool waited = false;
    for (int i = 0; i < (MODE == MODE_TM ? (n_my > 0 ? 1 : 0) : n_my); ++i) {
      const TileInfo ti = tile_info<MODE>(a, blockIdx.x + i * n_cta);
      if (ti.g != w_group) {  // (TM: once)
        if (w_loads > 0 && !mbar_wait(w_empty, (w_loads - 1) & 1, abort_flag, a.err)) break;
        const int wsel = MODE == MODE_SEQ ? ti.g : layer;
        if (lane == 0) {
          mbar_expect_tx(w_full, kW13Bytes + kW2Bytes);
          for (int c = 0; c < kChunks; ++c)
            for (int kb = 0; kb < 2; ++kb)
              tma_load_2d(sW13 + c * 65536 + kb * 32768, &tmW13, w_full, kb * 64, wsel * 2 * kHid + c * 256);
          for (int kb = 0; kb < 4; ++kb) tma_load_2d(sW2 + kb * 16384, &tmW2, w_full, kb * 64, wsel * kD);
        }
        w_group = ti.g;
        ++w_loads;
      }
      if (MODE == MODE_TM) break;  // the epilogue warps write the mixed activations into TMEM
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (i >= 1 && !mbar_wait(a_empty, (i - 1) & 1, abort_flag, a.err)) break;
      if (lane == 0) {
        mbar_expect_tx(a_full, kATile);
        tma_load_2d(sA, &tmA, a_full, 0, (int)ti.row0);
        tma_load_2d(sA + kATile / 2, &tmA, a_full, 64, (int)ti.row0);
      }
    }
    // (TM with the attention's block counters: every tile it publishes has waited for its own blocks)
    if (!waited && !(MODE == MODE_TM && a.attn_ready)) pdl_wait();
    if (MODE == MODE_TM && lane == 0 && a.ple_ready && layer == a.n_layers - 1) {
      // publish each tile once its 16 epilogue warps have written it: count it for its 128-row block, which the
      // PLE starts when all of the block's tiles are in (bounded wait, as every wait here)
      for (int i = 0; i < n_my; ++i) {
        const unsigned need = (unsigned)(kEpiWarps * (i + 1));
        const uint64_t t0 = global_timer_ns();
        bool ok = true;
        while (*reinterpret_cast<volatile unsigned*>(ydone) < need) {
          if (*abort_flag || global_timer_ns() - t0 > 1000000000ull) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
        if (!ok) break;
        __threadfence();
        atomicAdd(a.ple_ready + (blockIdx.x + i * n_cta) / 16, 1u);  // tile = 8 candidates, block = 16 tiles
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule and waits (it stays converged); lane 0 issues the MMAs and commits.
    // Order: up(0), then for every chunk k >= 1: up(k), down(k - 1); finally down(last). Chunk k is chunk
    // k % 2 of tile k / 2.
    constexpr uint32_t id_up = idesc_bf16(128, 256), id_dn = idesc_bf16(128, 128);
    const int total = n_my * kChunks;
    int w_group = -1, w_loads = 0;
    auto issue_up = [&](int cc) -> bool {
      const int i = cc / kChunks, c = cc % kChunks;
      if (c == 0) {
        const int g = tile_info<MODE>(a, blockIdx.x + i * n_cta).g;
        if (g != w_group) {
          if (!mbar_wait(w_full, w_loads & 1, abort_flag, a.err)) return false;
          w_group = g;
          ++w_loads;
        }
        if (!mbar_wait(a_full, i & 1, abort_flag, a.err)) return false;
      }
      if (cc >= 1 && !mbar_wait(up_empty, (cc - 1) & 1, abort_flag, a.err)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t aaddr = smem_u32(sA), w13 = smem_u32(sW13 + c * 65536);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16) {
          const uint64_t bd = sdesc_sw128(w13 + (k16 >> 2) * 32768 + (k16 & 3) * 32);
          if (MODE == MODE_SEQ)
            tc_mma(tbase + kColUp, sdesc_sw128(aaddr + (k16 >> 2) * (kATile / 2) + (k16 & 3) * 32), bd, id_up,
                   k16 != 0);
          else  // Mix(Z) in TMEM, buffer of this tile's parity: K = 16 bf16 per step = 8 columns
            tc_mma_ts(tbase + kColUp, tbase + kColA + (i & 1) * 64 + k16 * 8, bd, id_up, k16 != 0);
        }
        tc_commit(up_full);
        if (c == kChunks - 1) tc_commit(a_empty);
      }
      __syncwarp();
      return true;
    };
    auto issue_down = [&](int cc) -> bool {
      const int i = cc / kChunks, c = cc % kChunks;
      if (c == 0 && i >= 1 && !mbar_wait(dn_empty, (i - 1) & 1, abort_flag, a.err)) return false;
      if (!mbar_wait(hm_full, cc & 1, abort_flag, a.err)) return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t w2 = smem_u32(sW2 + (c * 2 + (k >> 2)) * 16384) + (k & 3) * 32;
          if (MODE == MODE_SEQ)
            tc_mma_ts(tbase + kColDown, tbase + kColHid + k * 8, sdesc_sw128(w2), id_dn, (c | k) != 0);
          else  // hidden chunk in shared memory: 2 K-blocks of [128 rows][64 units], 128B-swizzled
            tc_mma(tbase + kColDown, sdesc_sw128(smem_u32(sA) + (k >> 2) * 16384 + (k & 3) * 32), sdesc_sw128(w2),
                   id_dn, (c | k) != 0);
        }
        tc_commit(hm_empty);
        if (c == kChunks - 1) {
          tc_commit(dn_full);
          // the weights may be replaced once this tile's MMAs are done, if the next tile needs another group
          const int tile = blockIdx.x + i * n_cta, next = tile + n_cta;
          if (MODE == MODE_SEQ && next < n_tiles && tile_info<MODE>(a, next).g != tile_info<MODE>(a, tile).g)
            tc_commit(w_empty);
        }
      }
      __syncwarp();
      return true;
    };
    bool ok = total > 0 ? issue_up(0) : true;
    for (int k = 1; ok && k <= total; ++k) {
      if (k < total) {
        // a sequence tile of another group needs the weights reloaded, which needs every MMA of the previous
        // tile done: issue the pending down projection first
        const bool reload = MODE == MODE_SEQ && k % kChunks == 0 &&
                            tile_info<MODE>(a, blockIdx.x + (k / kChunks) * n_cta).g !=
                                tile_info<MODE>(a, blockIdx.x + (k / kChunks - 1) * n_cta).g;
        if (reload) {
          ok = issue_down(k - 1) && issue_up(k);
          continue;
        }
        ok = issue_up(k);
        if (!ok) break;
      }
      ok = issue_down(k - 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue (16 warps)
    // Warp (quarter q, group grp): TMEM lanes [32q, 32q + 32) -- tile rows -- and a quarter of the columns:
    // hidden units [32 grp, 32 grp + 32) of each chunk, output columns [32 grp, 32 grp + 32).
    const int q = warp & 3;               // TMEM lane quarter
    const int grp = (warp - 2) >> 2;      // column quarter
    const int rl = q * 32 + lane;         // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    // this warp's units within a chunk: up-buffer columns a = 128 (grp/2) + 32 (grp%2), g = a + 64
    const uint32_t col_a = 128 * (grp >> 1) + 32 * (grp & 1);
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
    // TM: each tile waits for the attention's groups of its 8 candidates (a 32-candidate block) instead of the
    // whole attention grid, when the attention counts them
    const bool by_block = MODE == MODE_TM && a.attn_ready != nullptr;
    if (!by_block) {
      pdl_wait();
      if (threadIdx.x == 64) CVR_TL_WAITED();
    }
    // true once the attention has written every group of the tile's block; block: wait (bounded) for it. Lane 0
    // reads the counter with acquire semantics and the warp barrier orders the other lanes' loads after it.
    auto z_ready = [&](int tile, bool block) -> bool {
      if (!by_block) return true;
      const unsigned need = (unsigned)(kG * (layer + 1));  // the counters sum over the layers
      int ready = 1;
      if (lane == 0) {
        if (block)
          wait_count(a.attn_ready + tile / 4, need, a.err);
        else
          ready = ld_acquire_u32(a.attn_ready + tile / 4) >= need;
      }
      ready = __shfl_sync(0xffffffffu, ready, 0);
      __syncwarp();
      return ready != 0;
    };
    // TM: this thread's 4 pieces Z[b][t][8j..8j+8) (tokens t = 4 grp.. of its column quarter), written into
    // TMEM lane (b, j) at columns 4t.., form the mixed activation row (b, j) (K slot t holds head j of token t)
    // that the up projection reads as its A operand; the same TMEM columns later give the residual back.
    const int bl = rl >> 4, j = rl & 15;
    auto load_z = [&](uint4* z, int tile) {
      // unconditional loads (rows past the batch read the last candidate and are never stored), so the
      // loads stay in flight until the registers are consumed; through L2, as the attention grid that wrote
      // the decoded tokens may still be running
      const int64_t bc = (int64_t)tile * (128 / kT) + bl;
      const int64_t bsrc = bc < a.B ? bc : a.B - 1;
#pragma unroll
      for (int tt = 0; tt < 4; ++tt)
        z[tt] = __ldcg(reinterpret_cast<const uint4*>(zin + bsrc * kYD + (grp * 4 + tt) * kD + j * 8));
    };
    auto store_a = [&](const uint4* z, int buf) {
      uint32_t w[16];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        w[4 * tt + 0] = z[tt].x;
        w[4 * tt + 1] = z[tt].y;
        w[4 * tt + 2] = z[tt].z;
        w[4 * tt + 3] = z[tt].w;
      }
      tmem_st16(tbase + lane_off + kColA + buf * 64 + grp * 16, w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full);
    };
    uint4 znext[4];
    int z_late = -1;  // TM: the next tile, when its block was not ready at the prefetch (loaded before it is stored)
    // chunk cc of tile i: silu(a) * g of this warp's 32 units, stored as the down projection's A operand
    auto chunk = [&](int i, int c, bool has_next) -> bool {
      const int cc = i * kChunks + c;
      if (!mbar_wait(up_full, cc & 1, abort_flag, a.err)) return false;
      tc_fence_after();
      // biases of these units: b1/b3 are stored like the W13 rows, 64 units of W1 then 64 of W3
      const float2* ba2 = reinterpret_cast<const float2*>(sb13 + (2 * c + (grp >> 1)) * 128 + 32 * (grp & 1));
      const float2* bg2 = ba2 + 32;
      uint32_t hp[16];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // two halves of 16 units (bounded register use)
        uint32_t ra[16], rg[16];
        tmem_ld16_nowait(tbase + lane_off + kColUp + col_a + 16 * hh, ra);
        tmem_ld16_nowait(tbase + lane_off + kColUp + col_a + 64 + 16 * hh, rg);
        tmem_ld_wait();
        if (hh == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(up_empty);
          // every up projection of this tile has completed: the next tile's activations may be written
          if (MODE == MODE_TM && c == kChunks - 1 && has_next) {
            if (z_late >= 0) {
              z_ready(z_late, true);
              load_z(znext, z_late);
              z_late = -1;
            }
            store_a(znext, (i + 1) & 1);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 bav = ba2[8 * hh + e], bgv = bg2[8 * hh + e];
          const uint64_t av = add_f32x2(f2pack(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1])),
                                        f2pack(bav.x, bav.y));
          const uint64_t gv = add_f32x2(f2pack(__uint_as_float(rg[2 * e]), __uint_as_float(rg[2 * e + 1])),
                                        f2pack(bgv.x, bgv.y));
          hp[8 * hh + e] = silu_half_mul_bf16x2(av, gv);
        }
      }
      if (cc >= 1 && !mbar_wait(hm_empty, (cc - 1) & 1, abort_flag, a.err)) return false;
      tc_fence_after();  // the previous chunk's down MMAs have finished reading the hidden buffer
      if (MODE == MODE_SEQ) {
        tmem_st16(tbase + lane_off + kColHid + grp * 16, hp);
        tmem_st_wait();
        tc_fence_before();
      } else {
        // units [32 grp, 32 grp + 32) = K-block grp/2, 16-byte chunks 4 (grp%2) .. +4 of row rl (swizzled)
        uint8_t* rowp = sA + (grp >> 1) * 16384 + rl * 128;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *reinterpret_cast<uint4*>(rowp + (((4 * (grp & 1) + m) ^ (rl & 7)) << 4)) =
              make_uint4(hp[4 * m], hp[4 * m + 1], hp[4 * m + 2], hp[4 * m + 3]);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(hm_full);
      return true;
    };
    // output epilogue of tile i: columns [32 grp, 32 grp + 32) of the down accumulator
    auto finish = [&](int i) -> bool {
      const TileInfo ti = tile_info<MODE>(a, blockIdx.x + i * n_cta);
      if (!mbar_wait(dn_full, i & 1, abort_flag, a.err)) return false;
      tc_fence_after();
      uint32_t rv[32];
      tmem_ld32_nowait(tbase + lane_off + kColDown + grp * 32, rv);
      if (MODE == MODE_SEQ) {
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dn_empty);
        const int64_t row = ti.row0 + rl;
        if (row < ti.rows_end) {
          const float* bb = sb2 + grp * 32;
          uint4* dst = reinterpret_cast<uint4*>(a.H + row * kD + grp * 32);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint4 p;
            uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int x = jj * 8 + 2 * e;
              pp[e] = pack_bf16(__uint_as_float(rv[x]) + bb[x], __uint_as_float(rv[x + 1]) + bb[x + 1]);
            }
            dst[jj] = p;
          }
        }
        return true;
      }
      // TM: this thread holds F(mixed row (b, j)); output token t of candidate b takes F[(b, j)][8t..8t+8) as
      // its head j (Revert), adds the residual Z[b][t][8j..8j+8) (back from this tile's activation columns)
      // and is RMS-normalised over its 128 dims, whose 16 heads live in the 16 lanes that share b. This warp
      // handles tokens [4 grp, 4 grp + 4).
      uint32_t zr[16];
      tmem_ld16_nowait(tbase + lane_off + kColA + (i & 1) * 64 + grp * 16, zr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dn_empty);
      const int64_t bcand = ti.row0 / kT + bl;
      const bool live = bcand < a.B;
      // x = F + b2 + Z for 4 tokens x 8 dims (packed pairs), then the 4 sums of squares reduce together
      uint64_t x2[4][4];
      float ss[4];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int t = grp * 4 + tt;
        const float2* bb = reinterpret_cast<const float2*>(sb2 + t * 8);
        const __nv_bfloat162* zp = reinterpret_cast<const __nv_bfloat162*>(&zr[4 * tt]);
        const uint32_t* v = &rv[tt * 8];
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
        for (int tt = 0; tt < 4; ++tt) ss[tt] += __shfl_xor_sync(0xffffffffu, ss[tt], o);
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const float inv = rsqrtf(ss[tt] * (1.f / kD) + a.eps);
        const uint64_t inv2 = f2pack(inv, inv);
        uint4 p;
        uint32_t* pp = reinterpret_cast<uint32_t*>(&p);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint64_t y = mul_f32x2(mul_f32x2(x2[tt][e], inv2), gj2[e]);
          pp[e] = pack_bf16(__uint_as_float((uint32_t)y), __uint_as_float((uint32_t)(y >> 32)));
        }
        if (live) *reinterpret_cast<uint4*>(yout + bcand * kYD + (grp * 4 + tt) * kD + j * 8) = p;
      }
      if (MODE == MODE_TM) {
        // this warp's part of the tile is written: count it in shared memory (the producer warp publishes whole
        // tiles to the PLE, so no epilogue warp waits on a device-scope fence)
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicAdd(ydone, 1u);
        }
      }
      return true;
    };
    if (MODE == MODE_TM && n_my > 0) {
      uint4 z0[4];
      z_ready(blockIdx.x, true);
      if (by_block && threadIdx.x == 64) CVR_TL_WAITED();
      load_z(z0, blockIdx.x);
      store_a(z0, 0);
    }
    // TM: the output epilogue of tile i runs after the first chunk of tile i + 1, while the tensor pipe works
    // on that tile's second up projection (the sequence encoder restages biases between groups, so it
    // finishes each tile before the next).
    constexpr bool kDefer = MODE == MODE_TM;
    for (int i = 0; i < n_my && ok; ++i) {
      const TileInfo ti = tile_info<MODE>(a, blockIdx.x + i * n_cta);
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
      const bool has_next = i + 1 < n_my;
      if (MODE == MODE_TM && has_next) {
        const int nt = blockIdx.x + (i + 1) * n_cta;
        if (z_ready(nt, false))
          load_z(znext, nt);
        else
          z_late = nt;
      }
      ok = chunk(i, 0, has_next);
      if (ok && kDefer && i >= 1) ok = finish(i - 1);
      if (ok) ok = chunk(i, 1, has_next);
      if (ok && !kDefer) ok = finish(i);
    }
    if (ok && kDefer && n_my > 0) finish(n_my - 1);
    if (MODE == MODE_SEQ) pdl_trigger();
  }
  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // (TM on the block counters: the kernel still completes only after the attention grid, so that whatever waits
  // for it waits for every earlier kernel too)
  if (MODE == MODE_TM && a.attn_ready && threadIdx.x == 0) pdl_wait();
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
  return launch_kernel(swiglu_mlp_kernel<MODE_SEQ>, dim3(grid), dim3(kThreads), kSmemBytes,
                       s, a.pdl != 0, a, tmXs, tmW13, tmW2, 0, n_tiles, grid, (const __nv_bfloat16*)nullptr,
                       (__nv_bfloat16*)nullptr);
}

cudaError_t launch_tm_mlp(const FwdArgs& a, int layer, const __nv_bfloat16* zin, __nv_bfloat16* yout,
                          const CUtensorMap& tmW13, const CUtensorMap& tmW2, cudaStream_t s) {
  const int n_tiles = (a.B + 7) / 8;  // 8 candidates x 16 mixed rows per tile
  const int grid = n_tiles < a.num_sms ? n_tiles : a.num_sms;
  // (the activation operand of the Token Mixer is written into TMEM by its epilogue warps: the first tensor map is
  // not used)
  return launch_kernel(swiglu_mlp_kernel<MODE_TM>, dim3(grid), dim3(kThreads), kSmemBytes, s, a.pdl != 0, a, tmW13,
                       tmW13, tmW2, layer, n_tiles, grid, zin, yout);
}

}  // namespace cvr
