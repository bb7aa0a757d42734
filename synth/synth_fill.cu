/* Device fill of seeded embedding tables: the same values as synth_table_rows() on the host,
 * written straight into device memory so that multi-GB tables never pass through the host. */
#include <cuda_runtime.h>
#include <stdint.h>

#include "cvr_synth.h"

__global__ void synth_fill_table_kernel(float* __restrict__ out, uint64_t seed, uint32_t table, uint64_t n,
                                        uint32_t dim, double scale) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t row = i / dim;
    const uint32_t col = (uint32_t)(i - row * dim);
    out[i] = synth_table_value(seed, table, row, col, dim, scale);
  }
}

/* Fills out[rows][dim] on `stream`. Returns a cudaError_t value (0 on success). */
extern "C" int synth_fill_table_device(float* out, uint64_t seed, uint32_t table, uint64_t rows, uint32_t dim,
                                       double scale, void* stream) {
  const uint64_t n = rows * (uint64_t)dim;
  if (n == 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  synth_fill_table_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, seed, table, n, dim, scale);
  return (int)cudaGetLastError();
}
