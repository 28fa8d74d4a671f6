// qdq.cu -- standalone dynamic per-tile FP8 E4M3 fake quantize-dequantize.
//
// "GDN state/W QAT foundation", "What does this PR do?": each tile has its own scalar
// scale amax / 448 with a zero guard, and a QDQ helper applies a supplied scale. One CTA
// per (leading index, tile): pass 1 reduces max|x| over the tile (max is exact, so the
// order does not matter), pass 2 rereads the tile (from L2) and writes E4M3(x / s) * s.
// HBM-bound: 4 bytes read + 4 bytes written per element.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kQdqThreads = 256;

// x and y may be the same buffer: each element is read and then written by one thread.
__global__ void __launch_bounds__(kQdqThreads)
tile_qdq_kernel(const float* x, float* y, float* __restrict__ scales, int rows, int cols,
                int tile_cols, int ntiles) {
  const int64_t blk = blockIdx.x;
  const int tile = (int)(blk % ntiles);
  const int64_t lead = blk / ntiles;
  const int j0 = tile * tile_cols;
  const int width = min(tile_cols, cols - j0);
  const float* xt = x + lead * (int64_t)rows * cols + j0;
  float* yt = y + lead * (int64_t)rows * cols + j0;
  const int n = rows * width;

  float amax = 0.0f;
  for (int e = threadIdx.x; e < n; e += kQdqThreads) {
    const int r = e / width, j = e - r * width;
    amax = fmaxf(amax, fabsf(xt[(int64_t)r * cols + j]));
  }
  __shared__ float red[kQdqThreads / 32];
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < kQdqThreads / 32 ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float s = qdq_scale(red[0]);
  if (scales && threadIdx.x == 0) scales[lead * ntiles + tile] = s;
  for (int e = threadIdx.x; e < n; e += kQdqThreads) {
    const int r = e / width, j = e - r * width;
    yt[(int64_t)r * cols + j] = qdq1(xt[(int64_t)r * cols + j], s);
  }
}

}  // namespace

cudaError_t launch_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int rows,
                            int cols, int tile_cols, cudaStream_t stream) {
  const int ntiles = (cols + tile_cols - 1) / tile_cols;
  const int64_t blocks = lead * ntiles;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  tile_qdq_kernel<<<(unsigned)blocks, kQdqThreads, 0, stream>>>(x, y, scales, rows, cols, tile_cols, ntiles);
  return cudaGetLastError();
}

}  // namespace gdn
