// tc_selftest.cu -- hardware check of the tensor-core operand layouts the chunked forward uses.
//
// One CTA of 128 threads computes D[M x N] = A[M x K] B[K x N] with tcgen05.mma from shared
// memory (A and B staged in the 128-byte-swizzled K-major or MN-major layout, bf16 or tf32
// values), accumulates in TMEM and writes every TMEM lane (128) x N columns back. The host
// compares with a CPU product. Every shared-memory access stays inside the 227 KB buffer and
// the only wait is bounded. Built into the test-only library, not the product library.
#include "../../fp8_state_qat_gb300/csrc/common.cuh"
#include "../../fp8_state_qat_gb300/csrc/tc_common.cuh"

namespace gdn {
namespace {

constexpr uint32_t kSmemBytes = 200 * 1024;   // + static smem stays under the 227 KB limit
constexpr uint32_t kBOffset = 64 * 1024;

__device__ void stage(unsigned char* base, const float* src, int rows, int cols, bool src_row_is_mn, int kind,
                      bool mn_major, int mn_extent, int k_extent) {
  // src is row-major [rows][cols]; logical operand element (mn, k)
  const int e = kind == tc::kKindTF32 ? 4 : 2;
  const int epr = 128 / e;   // elements per 128-byte row
  for (int idx = threadIdx.x; idx < rows * cols; idx += blockDim.x) {
    const int r = idx / cols, c = idx % cols;
    const int mn = src_row_is_mn ? r : c;
    const int k = src_row_is_mn ? c : r;
    uint32_t off;
    if (!mn_major) off = (uint32_t)(k / epr) * (uint32_t)(mn_extent * 128) + tc::sw128(mn, (k % epr) * e);
    else off = (uint32_t)(mn / epr) * (uint32_t)(k_extent * 128) + tc::sw128(k, (mn % epr) * e);
    const float x = src[idx];
    if (kind == tc::kKindTF32) *reinterpret_cast<float*>(base + off) = tc::to_tf32(x);
    else *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
  }
}

__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const float* A, const float* B, float* D, float* D2, int M, int N, int K, int kind, int a_mn,
                   int b_mn, int* status) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tmem_base_slot;
  const int warp = threadIdx.x >> 5;
  for (uint32_t i = threadIdx.x; i < kSmemBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  stage(smem, A, M, K, true, kind, a_mn, M, K);
  stage(smem + kBOffset, B, K, N, false, kind, b_mn, N, K);
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&mbar), 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_base_slot), 512);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_slot;
  if (threadIdx.x == 0) {
    const int kstep = kind == tc::kKindTF32 ? 8 : 16;
    const uint32_t idesc = tc::make_idesc(kind, M, N, a_mn != 0, b_mn != 0);
    const uint32_t a0 = tc::smem_u32(smem), b0 = tc::smem_u32(smem + kBOffset);
    for (int ks = 0; ks < K / kstep; ++ks) {
      uint64_t ad, bd;
      if (!a_mn) ad = tc::make_sdesc(a0 + (ks * 32 / 128) * (M * 128) + (ks * 32) % 128, 16, 1024);
      else ad = tc::make_sdesc(a0 + (ks * kstep / 8) * 1024, K * 128, 1024);
      if (!b_mn) bd = tc::make_sdesc(b0 + (ks * 32 / 128) * (N * 128) + (ks * 32) % 128, 16, 1024);
      else bd = tc::make_sdesc(b0 + (ks * kstep / 8) * 1024, K * 128, 1024);
      if (kind == tc::kKindTF32) tc::mma_tf32(tmem, ad, bd, idesc, ks > 0);
      else tc::mma_bf16(tmem, ad, bd, idesc, ks > 0);
    }
    tc::mma_commit(tc::smem_u32(&mbar));
  }
  const bool ok = tc::mbar_wait(tc::smem_u32(&mbar), 0, 1u << 22);   // its own limit: the test library lowers the default
  if (!ok && threadIdx.x == 0) atomicExch(status, 1);
  tc::tc_fence_after();
  if (ok) {
    const int lane = warp * 32 + (threadIdx.x & 31);
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tc::tmem_ld16(tc::tmem_addr(tmem, warp * 32, c0), v);
      tc::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) D[lane * N + c0 + j] = v[j];
    }
    if (D2) {   // the same accumulator read with the 16-lane two-half shape (split = N / 2); with
                // M = 128 also the upper 16 lanes of each quadrant (lane offset 16)
      const int t = threadIdx.x & 31;
      for (int lo16 = 0; lo16 < (M == 128 ? 32 : 16); lo16 += 16) {
        const int row = warp * 32 + lo16 + (t & 15);
        for (int c0 = 0; c0 < N / 2; c0 += 16) {
          float v[16];
          if (N == 128) tc::tmem_ld16x2<64>(tc::tmem_addr(tmem, warp * 32 + lo16, c0), v);
          else tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, warp * 32 + lo16, c0), v);
          tc::tmem_ld_wait();
          const int col = c0 + (t >> 4) * (N / 2);
#pragma unroll
          for (int j = 0; j < 16; ++j) D2[row * N + col + j] = v[j];
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace
}  // namespace gdn

// Internal: D [128 lanes x N] from A [M x K] and B [K x N] (device fp32, row-major) with the
// requested operand kind (0 bf16, 1 tf32) and majors; status (device int) set on a timeout.
// D2 (nullable): the accumulator read again with the 16x32bx2 TMEM load shape (M = 128: both
// 16-lane halves of every quadrant).
extern "C" int gdnqat_internal_tc_selftest(const float* A, const float* B, float* D, float* D2, int M, int N, int K,
                                           int kind, int a_mn, int b_mn, int* status, cudaStream_t stream) {
  if ((M != 64 && M != 128) || (N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
  cudaError_t e = cudaFuncSetAttribute(gdn::tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)gdn::kSmemBytes);
  if (e != cudaSuccess) return 2;
  gdn::tc_selftest_kernel<<<1, 128, gdn::kSmemBytes, stream>>>(A, B, D, D2, M, N, K, kind, a_mn, b_mn, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
