// tc_epilogue.cuh -- register/shared-memory helpers shared by the tensor-core chunk kernels.
#pragma once

#include "common.cuh"
#include "tc_common.cuh"

namespace gdn {

// bf16 pair packed in 32 bits (low half = first element)
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
// 8 consecutive values -> bf16 hi (exact rounding) and lo (residual), one 16-byte chunk each
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
    const float2 hf = unpack_bf16(h[i]);
    l[i] = pack_bf16(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ void st16(unsigned char* sm, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(sm + off) = v;
}
// E4M3 QDQ of a pair with the reciprocal of the scale: codes (as fp32) and dequantized values
__device__ __forceinline__ void qdq_pair(float a, float b, float rs, float s, float& ca, float& cb, float& qa,
                                         float& qb) {
  const __nv_fp8x2_e4m3 c(make_float2(__fmul_rn(a, rs), __fmul_rn(b, rs)));
  const float2 cf = static_cast<float2>(c);
  ca = cf.x;
  cb = cf.y;
  qa = __fmul_rn(cf.x, s);
  qb = __fmul_rn(cf.y, s);
}
// E4M3 codes (as fp32) of a pair scaled by the reciprocal of the tile scale
__device__ __forceinline__ void e4m3_codes2(float a, float b, float rs, float& ca, float& cb) {
  const __nv_fp8x2_e4m3 c(make_float2(__fmul_rn(a, rs), __fmul_rn(b, rs)));
  const float2 cf = static_cast<float2>(c);
  ca = cf.x;
  cb = cf.y;
}
__device__ __forceinline__ void ld32(uint32_t tmem, uint32_t lane0, uint32_t col, float* v) {
  tc::tmem_ld16(tc::tmem_addr(tmem, lane0, col), v);
  tc::tmem_ld16(tc::tmem_addr(tmem, lane0, col + 16), v + 16);
  tc::tmem_ld_wait();
}
__device__ __forceinline__ void st32(uint32_t tmem, uint32_t lane0, uint32_t col, const float* v) {
  tc::tmem_st16(tc::tmem_addr(tmem, lane0, col), v);
  tc::tmem_st16(tc::tmem_addr(tmem, lane0, col + 16), v + 16);
}
// max |v| over the 32 lanes of a warp (redux.sync, sm_100 family); NaN inputs do not win, as with fmaxf
__device__ __forceinline__ float warp_absmax(float v) {
  float r;
  asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// descriptor for `addr` advanced by `off` bytes (the start field is the low 14 bits, in 16-byte units)
__device__ __forceinline__ uint64_t dadv(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }


}  // namespace gdn
