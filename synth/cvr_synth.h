/* Seeded synthetic inputs for the CVR scoring workloads.
 *
 * This module produces the inputs that the scoring path and its CPU oracle
 * both consume: fp32 embedding tables, multi-hot bag ids and offsets,
 * behaviour-sequence ids and bf16-valued dense weights. It holds none of the
 * model's arithmetic. Every value is a pure function of (seed, stream, index)
 * through the SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), so a table row can be
 * evaluated on demand on the host or filled on the device with identical bits.
 *
 * Ids follow a Zipf law drawn by rejection-inversion (Hoermann & Derflinger,
 * "Rejection-inversion to generate variates from monotone discrete
 * distributions", ACM TOMACS 1996), which needs no CDF table, so 10^8-row
 * tables cost nothing to sample.
 */
#ifndef CVR_SYNTH_H
#define CVR_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Stream identifiers: each kind of input draws from its own stream. */
#define SYNTH_STREAM_TABLE 0x100u   /* + table index (0..15 fields, 16 = shared sequence table) */
#define SYNTH_STREAM_DENSE 0x1000u  /* + dense weight tensor index */
#define SYNTH_STREAM_BAGSIZE 0x2000u
#define SYNTH_STREAM_IDS 0x3000u    /* + field index */
#define SYNTH_STREAM_SEQ 0x4000u
#define SYNTH_STREAM_PERM 0x5000u   /* + table index: offset of the rank->row bijection */
#define SYNTH_STREAM_LENS 0x6000u   /* variable sequence lengths */

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ull

SYNTH_HD uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Counter-based hash of (seed, stream, index). */
SYNTH_HD uint64_t synth_hash(uint64_t seed, uint64_t stream, uint64_t index) {
  return synth_mix64(synth_mix64(seed + SYNTH_GAMMA * (stream + 1u)) + SYNTH_GAMMA * (index + 1u));
}

/* Embedding table entry T[table][row][col] = fp32(scale * (2u - 1)), u = 24 hash bits / 2^24.
 * Computed in double with one rounding to fp32, so host and device agree bit for bit. */
SYNTH_HD float synth_table_value(uint64_t seed, uint32_t table, uint64_t row, uint32_t col, uint32_t dim,
                                 double scale) {
  const uint64_t h = synth_hash(seed, SYNTH_STREAM_TABLE + table, row * (uint64_t)dim + col);
  const double u = (double)(h >> 40) * (1.0 / 16777216.0);
  return (float)(scale * (2.0 * u - 1.0));
}

/* ---- host-side generators (cvr_synth.c) ---- */

/* Fill rows [row0, row0+nrows) of a table, row-major [nrows][dim]. */
void synth_table_rows(uint64_t seed, uint32_t table, uint64_t row0, uint64_t nrows, uint32_t dim, double scale,
                      float* out);

/* n values uniform in [-bound, bound), each rounded to the nearest bf16 (ties to even) and stored as fp32. */
void synth_uniform_bf16(uint64_t seed, uint32_t stream, int64_t n, double bound, float* out);

/* One Zipf(s) rank in 1..n, drawn from the uniforms hash(seed, stream, (index << 6) + attempt). */
int64_t synth_zipf_rank(uint64_t seed, uint32_t stream, uint64_t index, int64_t n, double s);

/* Rank -> row bijection: row = ((rank-1) * P + K) mod rows, P = 1000003 (prime, coprime with every
 * table size used here), K drawn per table. Scatters the hot ranks across the table. */
int64_t synth_rank_to_row(uint64_t seed, uint32_t table, int64_t rank, int64_t rows);

/* Multi-hot bags. Bags are numbered 0..n_bags-1; bag i draws its size uniformly in [min_size, max_size]
 * and its ids from table field_of_bag[i] (rows[field] rows, Zipf exponent s).
 * offsets[n_bags+1] is written as a CSR prefix; ids must hold offsets[n_bags] entries
 * (call once with ids == NULL to get the total through offsets). */
void synth_bags(uint64_t seed, int64_t n_bags, const int32_t* field_of_bag, const int64_t* rows, int32_t min_size,
                int32_t max_size, double s, int64_t* offsets, int64_t* ids);

/* Sequence ids [n_req][sum_len][cols], every id a Zipf(s) row of the shared table (table index 16). */
void synth_seq_ids(uint64_t seed, int64_t n_req, int64_t sum_len, int32_t cols, int64_t rows, double s, int64_t* ids);

/* Variable sequence lengths [n_req][n_groups]: lens[r][g] uniform in [min_len, seq_len[g]]. */
void synth_seq_lens(uint64_t seed, int64_t n_req, int32_t n_groups, const int32_t* seq_len, int32_t min_len,
                    int32_t* lens);

#ifdef __cplusplus
}
#endif
#endif
