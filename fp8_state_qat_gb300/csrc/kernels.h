// kernels.h -- internal launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

struct ChunkProblem {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;   // device cu_seqlens or null
  float* o;
  float* hT;
  int B, T, N, Hqk, Hv, dk, dv;
  float scale;
  int state_qdq, w_qdq, kda;
};

cudaError_t launch_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int rows, int cols,
                            int tile_cols, cudaStream_t stream);

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, float* o, int N, int Hqk, int Hv, int dk, int dv, float scale,
                          int state_qdq, int kda, cudaStream_t stream);

// Fused tensor-core chunked forward (tcgen05 + TMA), dk = 128, GDN. status: device int,
// set to nonzero when a bounded wait gives up.
bool chunk_tc_supported(const ChunkProblem& p);
cudaError_t launch_chunk_tc(const ChunkProblem& p, int* status, cudaStream_t stream);

// TMA descriptor of a head-last bf16 tensor [tokens, heads, D] with 64 x 1 x 64 boxes
// (128-byte swizzle). Host only; false when the driver entry point is unavailable.
bool make_bf16_map(CUtensorMap* map, const void* base, int D, int heads, int64_t tokens);

// Per-CTA fp32 chunked forward on CUDA cores: one CTA per (sequence, head, 64-column
// value slab). Used for shapes and variants the tensor-core path does not take.
cudaError_t launch_chunk_simt(const ChunkProblem& p, cudaStream_t stream);

}  // namespace gdn
