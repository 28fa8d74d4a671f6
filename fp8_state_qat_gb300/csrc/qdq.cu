// qdq.cu -- standalone dynamic per-tile FP8 E4M3 fake quantize-dequantize.
//
// "GDN state/W QAT foundation", "What does this PR do?": one scale per tile, amax / 448 (1 for
// an all-zero tile); the page's helper applies a scale it is given. One CTA
// per tile: max|x| over the tile (max is exact, so the order does not matter), then
// E4M3(x / s) * s with x / s correctly rounded. HBM-bound: 4 bytes read + 4 bytes written per
// element. Three launch forms, by shape: whole rows of a leading index per CTA (state and W
// tiles: every warp reads contiguous rows, measured 0.91 of the copy bandwidth against 0.65 for
// one CTA per 64-column tile), one register-resident tile per CTA, or a general two-pass form
// that rereads the tile from L2.
#include "common.cuh"
#include "kernels.h"
#include "tc_epilogue.cuh"

namespace gdn {
namespace {

constexpr int kQdqThreads = 256;
constexpr int kQdqRegF4 = 8;   // float4 per thread on the register path: tiles up to 8192 elements

__device__ __forceinline__ float2 qdq_exact2(float a, float b, float s, float r, bool fast) {
  const float2 y = fast ? quotient2(make_float2(a, b), make_float2(-s, -s), make_float2(r, r))
                        : make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
  const __nv_fp8x2_e4m3 c(y);          // cvt.rn.satfinite.e4m3x2.f32
  return __fmul2_rn(static_cast<float2>(c), make_float2(s, s));
}

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kQdqThreads / 32 ? red[threadIdx.x] : 0.0f;
    w = warp_max(w);
    if (threadIdx.x == 0) red[0] = w;
  }
  __syncthreads();
  return red[0];
}

// Register path: one CTA per (leading index, tile) with the tile (rows x width <= 8192, width a
// multiple of 4, 16-byte aligned rows) read once into registers as float4, reduced, then
// quantized from registers. x and y may be the same buffer.
__global__ void __launch_bounds__(kQdqThreads)
tile_qdq_reg_kernel(const float* x, float* y, float* __restrict__ scales, int rows, int cols, int tile_cols,
                    int ntiles) {
  const int64_t blk = blockIdx.x;
  const int tile = (int)(blk % ntiles);
  const int64_t lead = blk / ntiles;
  const int j0 = tile * tile_cols;
  const int width = min(tile_cols, cols - j0);
  const int w4 = width >> 2, n4 = rows * w4;
  const float* xt = x + lead * (int64_t)rows * cols + j0;
  float* yt = y + lead * (int64_t)rows * cols + j0;
  float4 v[kQdqRegF4];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kQdqRegF4; ++i) {
    const int u = threadIdx.x + i * kQdqThreads;
    if (u < n4) {
      const int r = u / w4, c4 = u - r * w4;
      v[i] = __ldcs(reinterpret_cast<const float4*>(xt + (int64_t)r * cols + 4 * c4));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
  }
  __shared__ float red[kQdqThreads / 32];
  const float s = qdq_scale(block_max(amax, red));
  if (scales && threadIdx.x == 0) scales[lead * ntiles + tile] = s;
  const bool fast = s >= 1.17549435e-38f;   // normal scale: the reciprocal path is exact
  const float rcp = __frcp_rn(s);
#pragma unroll
  for (int i = 0; i < kQdqRegF4; ++i) {
    const int u = threadIdx.x + i * kQdqThreads;
    if (u < n4) {
      const int r = u / w4, c4 = u - r * w4;
      const float2 a = qdq_exact2(v[i].x, v[i].y, s, rcp, fast), b = qdq_exact2(v[i].z, v[i].w, s, rcp, fast);
      __stcs(reinterpret_cast<float4*>(yt + (int64_t)r * cols + 4 * c4), make_float4(a.x, a.y, b.x, b.y));
    }
  }
}

// Whole-row path: one CTA of 512 threads per leading index; cols / 4 divides 512, so each thread
// always touches the same four columns (one tile), and a warp reads whole rows.
constexpr int kLeadThreads = 512;
__global__ void __launch_bounds__(kLeadThreads)
tile_qdq_lead_kernel(const float* x, float* y, float* __restrict__ scales, int rows, int cols, int tile_cols,
                     int ntiles) {
  constexpr int F4 = 8;
  __shared__ float red[kLeadThreads / 32][4];
  const int64_t lead = blockIdx.x;
  const int c4n = cols >> 2, n4 = rows * c4n;
  const int c4 = threadIdx.x % c4n;
  const int mytile = (4 * c4) / tile_cols;
  const float* xl = x + lead * (int64_t)rows * cols;
  float* yl = y + lead * (int64_t)rows * cols;
  float4 v[F4];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < F4; ++i) {
    const int u = threadIdx.x + i * kLeadThreads;
    if (u < n4) {
      v[i] = *reinterpret_cast<const float4*>(xl + 4 * (int64_t)u);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
  }
  // per-tile max: a warp covers 128 consecutive columns, so at most 3 tiles of >= 64 columns
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = (4 * ((warp * 32) % c4n)) / tile_cols;   // first tile this warp touches
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m = (mytile == t0 + k) ? amax : 0.f;
    m = warp_max(m);
    if (lane == 0) red[warp][k] = m;
  }
  __syncthreads();
  float m = 0.f;
  for (int w = 0; w < kLeadThreads / 32; ++w) {
    const int tw = (4 * ((w * 32) % c4n)) / tile_cols;
    const int k = mytile - tw;
    if (k >= 0 && k < 4) m = fmaxf(m, red[w][k]);
  }
  const float s = qdq_scale(m);
  if (scales && (threadIdx.x % c4n) * 4 == mytile * tile_cols && threadIdx.x < c4n) scales[lead * ntiles + mytile] = s;
  const bool fast = s >= 1.17549435e-38f;
  const float rcp = __frcp_rn(s);
#pragma unroll
  for (int i = 0; i < F4; ++i) {
    const int u = threadIdx.x + i * kLeadThreads;
    if (u < n4) {
      const float2 a = qdq_exact2(v[i].x, v[i].y, s, rcp, fast), b = qdq_exact2(v[i].z, v[i].w, s, rcp, fast);
      *reinterpret_cast<float4*>(yl + 4 * (int64_t)u) = make_float4(a.x, a.y, b.x, b.y);
    }
  }
}

// General path: any shape; pass 1 reduces max|x| over the tile, pass 2 rereads it (from L2).
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
  const float s = qdq_scale(block_max(amax, red));
  if (scales && threadIdx.x == 0) scales[lead * ntiles + tile] = s;
  const bool fast = s >= 1.17549435e-38f;
  const float rcp = __frcp_rn(s);
  for (int e = threadIdx.x; e < n; e += kQdqThreads) {
    const int r = e / width, j = e - r * width;
    yt[(int64_t)r * cols + j] = qdq_exact2(xt[(int64_t)r * cols + j], 0.0f, s, rcp, fast).x;
  }
}

// INT8 block codec (page "Torch GDN/KDA decode QAT with INT8 recurrent state", summary: one
// scale per 32-value block of the state): one warp per block of one row (block_cols consecutive
// columns, the last block of a row narrower), amax = max |x| (redux), s = amax / 127 (IEEE
// divide, zero guard), c = nearest integer to x / s (ties to even) within [-127, 127], y = c * s.
// x / s is the correctly rounded quotient (common.cuh's corrected reciprocal for normal s, else an IEEE divide; a
// subnormal quotient rounds to 0 either way), so the result is bit-for-bit the fp32 definition.
// HBM-bound: 4 bytes read + 4 written per element; with 32-column blocks a warp moves 128
// contiguous bytes each way.
constexpr int kInt8Warps = 8;
__global__ void __launch_bounds__(kInt8Warps * 32)
int8_block_qdq_kernel(const float* x, float* y, float* __restrict__ scales, int64_t rows, int cols, int block_cols,
                      int nb) {
  const int lane = threadIdx.x & 31;
  const int64_t total = rows * nb;
  for (int64_t blk = (int64_t)blockIdx.x * kInt8Warps + (threadIdx.x >> 5); blk < total;
       blk += (int64_t)gridDim.x * kInt8Warps) {
    const int64_t r = blk / nb;
    const int b = (int)(blk - r * nb);
    const int j0 = b * block_cols, n = min(block_cols, cols - j0);
    const float* xb = x + r * cols + j0;
    float* yb = y + r * cols + j0;
    // blocks of up to 32 columns: one element per lane, held in a register between the passes
    const float v0 = lane < n ? __ldcs(xb + lane) : 0.0f;
    float amax = fabsf(v0);
    for (int j = lane + 32; j < n; j += 32) amax = fmaxf(amax, fabsf(xb[j]));
    amax = warp_absmax(amax);
    const float s = int8_scale(amax);
    if (scales && lane == 0) scales[blk] = s;
    const bool fast = s >= 1.17549435e-38f;
    const float rs = fast ? __frcp_rn(s) : 0.0f;
    for (int j = lane; j < n; j += 32) {
      const float v = j == lane ? v0 : xb[j];
      const float q = fast ? quotient(v, s, rs) : __fdiv_rn(v, s);
      const float c = fminf(fmaxf(rintf(q), -kInt8Max), kInt8Max);
      __stcs(yb + j, __fmul_rn(c, s));
    }
  }
}

// The same codec for 32-column blocks of 16-byte aligned rows (the state codec's shape): a lane
// holds one float4, 8 lanes one block, and each warp keeps kInt8Unroll x 512 bytes in flight, so
// the copy runs at HBM speed instead of one 128-byte block per warp at a time.
constexpr int kInt8Unroll = 4;
__global__ void __launch_bounds__(kInt8Warps * 32)
int8_block32_qdq_kernel(const float4* x, float4* y, float* __restrict__ scales, int64_t nblk) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kInt8Warps;
  // a warp step covers kInt8Unroll x 4 consecutive blocks (block = 8 float4)
  for (int64_t base = ((int64_t)blockIdx.x * kInt8Warps + (threadIdx.x >> 5)) * (4 * kInt8Unroll); base < nblk;
       base += warps * 4 * kInt8Unroll) {
    float4 v[kInt8Unroll];
#pragma unroll
    for (int u = 0; u < kInt8Unroll; ++u) {
      const int64_t blk = base + 4 * u + (lane >> 3);
      v[u] = blk < nblk ? __ldcs(x + blk * 8 + (lane & 7)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kInt8Unroll; ++u) {
      const int64_t blk = base + 4 * u + (lane >> 3);
      float m = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      if (blk >= nblk) continue;
      const float s = int8_scale(m);
      if (scales && (lane & 7) == 0) scales[blk] = s;
      const bool fast = s >= 1.17549435e-38f;
      const float rs = fast ? __frcp_rn(s) : 0.0f;
      auto q2 = [&](float a, float b) {   // codes: nearest integer of the quotient within +-127
        const float2 t = fast ? quotient2(make_float2(a, b), make_float2(-s, -s), make_float2(rs, rs))
                              : make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
        const float2 c = make_float2(fminf(fmaxf(rintf(t.x), -kInt8Max), kInt8Max),
                                     fminf(fmaxf(rintf(t.y), -kInt8Max), kInt8Max));
        return __fmul2_rn(c, make_float2(s, s));
      };
      const float2 lo = q2(v[u].x, v[u].y), hi = q2(v[u].z, v[u].w);
      __stcs(y + blk * 8 + (lane & 7), make_float4(lo.x, lo.y, hi.x, hi.y));
    }
  }
}

}  // namespace

cudaError_t launch_int8_block_qdq(const float* x, float* y, float* scales, int64_t rows, int cols, int block_cols,
                                  cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int nb = (cols + block_cols - 1) / block_cols;
  if (block_cols == 32 && cols % 32 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
    const int64_t nblk = rows * nb, per_warp = 4 * kInt8Unroll;
    int64_t grid = (nblk + per_warp * kInt8Warps - 1) / (per_warp * kInt8Warps);
    if (grid > 152 * 16) grid = 152 * 16;   // grid-stride: 16 CTAs of 8 warps per SM at most
    int8_block32_qdq_kernel<<<(unsigned)grid, kInt8Warps * 32, 0, stream>>>(
        reinterpret_cast<const float4*>(x), reinterpret_cast<float4*>(y), scales, nblk);
    return cudaGetLastError();
  }
  const int64_t warps = rows * nb;
  int64_t grid = (warps + kInt8Warps - 1) / kInt8Warps;
  if (grid > 152 * 64) grid = 152 * 64;   // grid-stride beyond 64 resident-sized waves of CTAs
  int8_block_qdq_kernel<<<(unsigned)grid, kInt8Warps * 32, 0, stream>>>(x, y, scales, rows, cols, block_cols, nb);
  return cudaGetLastError();
}

cudaError_t launch_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int rows,
                            int cols, int tile_cols, cudaStream_t stream) {
  const int ntiles = (cols + tile_cols - 1) / tile_cols;
  const int64_t blocks = lead * ntiles;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // the register path needs every tile (the last one too) to be float4 rows that fit in registers
  const int last = cols - (ntiles - 1) * tile_cols;
  const bool reg = tile_cols % 4 == 0 && cols % 4 == 0 && last % 4 == 0 &&
                   (int64_t)rows * tile_cols <= (int64_t)kQdqThreads * kQdqRegF4 * 4 &&
                   (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  const bool whole = cols % 4 == 0 && tile_cols % 4 == 0 && tile_cols >= 64 && (cols % tile_cols == 0) && kLeadThreads % (cols / 4) == 0 &&
                     (int64_t)rows * cols <= (int64_t)kLeadThreads * 8 * 4 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  if (whole)
    tile_qdq_lead_kernel<<<(unsigned)lead, kLeadThreads, 0, stream>>>(x, y, scales, rows, cols, tile_cols, ntiles);
  else if (reg)
    tile_qdq_reg_kernel<<<(unsigned)blocks, kQdqThreads, 0, stream>>>(x, y, scales, rows, cols, tile_cols, ntiles);
  else
    tile_qdq_kernel<<<(unsigned)blocks, kQdqThreads, 0, stream>>>(x, y, scales, rows, cols, tile_cols, ntiles);
  return cudaGetLastError();
}

}  // namespace gdn
