/* Host-side seeded input generators; see cvr_synth.h for the definitions. */
#include "cvr_synth.h"

#include <math.h>
#include <string.h>

void synth_table_rows(uint64_t seed, uint32_t table, uint64_t row0, uint64_t nrows, uint32_t dim, double scale,
                      float* out) {
  for (uint64_t r = 0; r < nrows; ++r)
    for (uint32_t c = 0; c < dim; ++c) out[r * dim + c] = synth_table_value(seed, table, row0 + r, c, dim, scale);
}

static float round_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest, ties to even (no NaN/Inf are generated) */
  u &= 0xFFFF0000u;
  memcpy(&x, &u, 4);
  return x;
}

void synth_uniform_bf16(uint64_t seed, uint32_t stream, int64_t n, double bound, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t h = synth_hash(seed, stream, (uint64_t)i);
    const double u = (double)(h >> 11) * (1.0 / 9007199254740992.0); /* 53 bits -> [0,1) */
    out[i] = round_bf16((float)(bound * (2.0 * u - 1.0)));
  }
}

static double unit_open(uint64_t seed, uint32_t stream, uint64_t index) {
  /* uniform in (0,1): 53 hash bits, offset by half an ulp so 0 is never returned */
  const uint64_t h = synth_hash(seed, stream, index);
  return ((double)(h >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Rejection-inversion for the Zipf law P(k) ~ k^-s on {1..n} (s > 0, s != 1).
 * h(x) = x^-s is the hat density; Hint(x) = (x^(1-s) - 1)/(1-s) is its integral and
 * Hinv its inverse. A continuous variate X is drawn by inverting Hint over
 * [Hint(1.5) - 1, Hint(n + 0.5)], rounded to k, and accepted when it falls under the
 * histogram bar of k (or inside the precomputed squeeze). */
static double zipf_Hint(double x, double one_minus_s) {
  const double lx = log(x);
  return expm1(one_minus_s * lx) / one_minus_s;
}
static double zipf_Hinv(double y, double one_minus_s) { return exp(log1p(one_minus_s * y) / one_minus_s); }
static double zipf_h(double x, double s) { return exp(-s * log(x)); }

int64_t synth_zipf_rank(uint64_t seed, uint32_t stream, uint64_t index, int64_t n, double s) {
  if (n <= 1) return 1;
  const double a = 1.0 - s;
  const double h_lo = zipf_Hint(1.5, a) - 1.0;
  const double h_hi = zipf_Hint((double)n + 0.5, a);
  const double squeeze = 2.0 - zipf_Hinv(zipf_Hint(2.5, a) - zipf_h(2.0, s), a);
  int64_t k = 1;
  for (uint64_t attempt = 0; attempt < 64; ++attempt) {
    const double u = h_hi + unit_open(seed, stream, (index << 6) + attempt) * (h_lo - h_hi);
    const double x = zipf_Hinv(u, a);
    k = (int64_t)(x + 0.5);
    if (k < 1) k = 1;
    if (k > n) k = n;
    if ((double)k - x <= squeeze || u >= zipf_Hint((double)k + 0.5, a) - zipf_h((double)k, s)) return k;
  }
  return k;
}

int64_t synth_rank_to_row(uint64_t seed, uint32_t table, int64_t rank, int64_t rows) {
  const uint64_t K = synth_hash(seed, SYNTH_STREAM_PERM + table, 0) % (uint64_t)rows;
  const uint64_t P = 1000003ull;
  return (int64_t)((((uint64_t)(rank - 1) % (uint64_t)rows) * (P % (uint64_t)rows) + K) % (uint64_t)rows);
}

void synth_bags(uint64_t seed, int64_t n_bags, const int32_t* field_of_bag, const int64_t* rows, int32_t min_size,
                int32_t max_size, double s, int64_t* offsets, int64_t* ids) {
  const uint64_t span = (uint64_t)(max_size - min_size + 1);
  offsets[0] = 0;
  for (int64_t i = 0; i < n_bags; ++i) {
    const int64_t size = min_size + (int64_t)((synth_hash(seed, SYNTH_STREAM_BAGSIZE, (uint64_t)i) >> 32) % span);
    offsets[i + 1] = offsets[i] + size;
    if (!ids) continue;
    const int32_t f = field_of_bag[i];
    for (int64_t p = 0; p < size; ++p) {
      const int64_t rank = synth_zipf_rank(seed, SYNTH_STREAM_IDS + (uint32_t)f, (uint64_t)(i * 64 + p), rows[f], s);
      ids[offsets[i] + p] = synth_rank_to_row(seed, (uint32_t)f, rank, rows[f]);
    }
  }
}

void synth_seq_ids(uint64_t seed, int64_t n_req, int64_t sum_len, int32_t cols, int64_t rows, double s, int64_t* ids) {
  const int64_t n = n_req * sum_len * cols;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t rank = synth_zipf_rank(seed, SYNTH_STREAM_SEQ, (uint64_t)i, rows, s);
    ids[i] = synth_rank_to_row(seed, 16u, rank, rows);
  }
}

void synth_seq_lens(uint64_t seed, int64_t n_req, int32_t n_groups, const int32_t* seq_len, int32_t min_len,
                    int32_t* lens) {
  for (int64_t r = 0; r < n_req; ++r)
    for (int32_t g = 0; g < n_groups; ++g) {
      const int32_t lo = min_len < seq_len[g] ? min_len : seq_len[g];
      const uint64_t span = (uint64_t)(seq_len[g] - lo) + 1u;
      lens[r * n_groups + g] = lo + (int32_t)(synth_hash(seed, SYNTH_STREAM_LENS, (uint64_t)(r * n_groups + g)) % span);
    }
}
