// common.cuh -- device helpers shared by the kernels of libgdnqat (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdnqat.h"

namespace gdn {

constexpr int kChunk = 64;          // chunk length fixed by the method ("GDN state/W QAT foundation")
constexpr int kStateTileCols = 64;  // state QDQ tile: all dk rows x 64 value columns (same page)
constexpr float kE4M3Max = 448.0f;  // largest finite E4M3 (fn) magnitude

// Scale of one QDQ tile from its amax: amax / 448 with the zero guard (0 -> 1), in fp32 with
// round-to-nearest division. The quotient is formed as the rounded reciprocal of 448 plus two FMA
// corrections (see quotient() below: correctly rounded for a normal quotient), the IEEE divide
// below 1e-30; equal to __fdiv_rn(amax, 448) for every non-negative finite amax (checked
// exhaustively on the GPU by the test suite).
__device__ __forceinline__ float qdq_scale(float amax) {
  float s;
  if (amax >= 1.0e-30f) {
    constexpr float r = 1.0f / kE4M3Max;
    const float q0 = __fmul_rn(amax, r);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, kE4M3Max, amax), r, q0);
    s = __fmaf_rn(__fmaf_rn(-q1, kE4M3Max, amax), r, q1);
  } else {
    s = __fdiv_rn(amax, kE4M3Max);
  }
  return s == 0.0f ? 1.0f : s;
}

// Two elements x -> E4M3(x / s) * s. The divide is IEEE round-to-nearest; the E4M3
// conversion is the hardware round-to-nearest-even with saturation to +-448; the
// product back is one fp32 multiply. The E4M3 value is exact in fp32.
__device__ __forceinline__ float2 qdq2(float a, float b, float s) {
  const float2 y = make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
  const __nv_fp8x2_e4m3 c(y);          // cvt.rn.satfinite.e4m3x2.f32
  const float2 cf = static_cast<float2>(c);
  return make_float2(__fmul_rn(cf.x, s), __fmul_rn(cf.y, s));
}

__device__ __forceinline__ float qdq1(float a, float s) {
  return qdq2(a, 0.0f, s).x;
}

// fl32(x / s) for the standalone QDQ ops from the round-to-nearest reciprocal r of s and two
// FMA corrections. q0 = fl32(x r) is within two ulps of x / s, so q1 = fl32(q0 + fl32(x - q0 s) r)
// misses x / s by far less than an ulp and is faithful (one of the two floats around x / s);
// its residual x - q1 s is exact in one FMA, and by Markstein's theorem (a faithful quotient, r
// correctly rounded) q2 = fl32(q1 + (x - q1 s) r) is the correctly rounded quotient, barring a
// subnormal quotient. A single correction is not enough in general: q0 need not be faithful.
// Callers use it only for normal s (then 1 / s is finite and normal); a subnormal quotient is
// below 2^-126, far under half the smallest E4M3 subnormal, so its code is 0 either way -- the
// E4M3 code of every element is the one the IEEE division gives (checked exhaustively over
// significands on the GPU against the IEEE divide by the test suite).
// The corrections turn -0 into +0; x / s with s > 0 always has the sign of x, so it is copied back.
__device__ __forceinline__ float quotient(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x), r, q0);
  return copysignf(__fmaf_rn(__fmaf_rn(-q1, s, x), r, q1), x);
}
// The same for two elements with the paired fp32 instructions (each component rounded as the
// scalar form rounds it): ns2 = (-s, -s), r2 = (r, r).
__device__ __forceinline__ float2 quotient2(float2 x, float2 ns2, float2 r2) {
  const float2 q0 = __fmul2_rn(x, r2);
  const float2 q1 = __ffma2_rn(__ffma2_rn(q0, ns2, x), r2, q0);
  const float2 q2 = __ffma2_rn(__ffma2_rn(q1, ns2, x), r2, q1);
  return make_float2(copysignf(q2.x, x.x), copysignf(q2.y, x.y));
}
// ---- INT8 block codec of the state (page "Torch GDN/KDA decode QAT with INT8 recurrent state",
// its summary): signed INT8 codes, one scale per block of 32; a block is 32 consecutive value
// columns of one key row; scale = amax / 127 (IEEE divide) with the zero guard; code = nearest
// integer to x / scale, ties to even, within [-127, 127]; value = code * scale.
constexpr int kInt8BlockCols = 32;
constexpr float kInt8Max = 127.0f;
// fl32(amax / 127) by Markstein's correction: with r = RN(1 / 127), q0 = RN(amax r) and the
// exact residual e = amax - q0 127 (one FMA), RN(q0 + e r) is the correctly rounded quotient
// whenever it is a normal number; smaller amax take the IEEE divide.
__device__ __forceinline__ float int8_scale(float amax) {
  constexpr float r = 1.0f / 127.0f;
  float s;
  if (amax >= 1.0e-30f) {
    const float q0 = __fmul_rn(amax, r);
    s = __fmaf_rn(__fmaf_rn(-q0, kInt8Max, amax), r, q0);
  } else {
    s = __fdiv_rn(amax, kInt8Max);
  }
  return s == 0.0f ? 1.0f : s;
}
// Fused form: x times the round-to-nearest reciprocal r of the scale. |x| <= amax keeps |x r|
// below 127 (1 + 2^-21), whose nearest integer lies within +-127, so no clamp is needed.
__device__ __forceinline__ float int8_qdq_rcp(float x, float r, float s) { return __fmul_rn(rintf(__fmul_rn(x, r)), s); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 bf16 (16 bytes) -> 8 fp32
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* p, float* out) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

}  // namespace gdn
