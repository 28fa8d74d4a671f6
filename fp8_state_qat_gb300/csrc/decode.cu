// decode.cu -- single-token decode step with per-token state QDQ (E4M3 tiles or INT8 blocks).
//
// Order per (sequence, head), as stated on "Torch GDN/KDA decode QAT with INT8 recurrent
// state" ("Megatron-Core QAT/QAD workflow", step 3) and "Add experimental GDN/KDA decode and
// replay QAT" (per-token FP8 state writes): read the stored state, S' = a S (KDA: row c scaled
// by a[c]), d = b (v - S'^T k), S = S' + k d^T, o = scale S^T q from the updated state, then
// per-tile QDQ (all dk rows x 64 value columns, scale amax / 448, zero guard) and store; with
// the INT8 codec ("Torch GDN/KDA decode QAT with INT8 recurrent state": dynamic INT8 block-32
// state recipes) one scale per key row and 32 value columns, amax / 127.
//
// HBM-bound: per (sequence, head) the state is read once and written once (2 * 4 dk dv
// bytes) plus the token's q, k, v, g, beta and o. The QDQ multiplies by the reciprocal of the
// tile scale (as the chunk kernels do) rather than dividing each element: an IEEE fp32 divide
// per element made the kernel issue-bound (0.77 -> 1.03 of the measured copy bandwidth). One CTA per (sequence, head); warp w
// owns value columns [16 w, 16 w + 16); lane = 4 * rg + cg holds rows rg, rg + 8, ... and
// the 4 columns 16 w + 4 cg .. + 3 as float4 registers, so the state moves with 16-byte
// coalesced accesses and both dk-reductions are 3-level xor shuffles (lane bits 2..4) in
// a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

template <int DK, int DV, bool KDA>
__global__ void __launch_bounds__(DV * 2, (DV <= 128 ? 2 : 1))
decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
              const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
              const float* __restrict__ beta, float* __restrict__ state, float* __restrict__ o,
              int Hqk, int Hv, float scale, int state_qdq) {
  constexpr int NW = DV / 16;      // warps per CTA
  constexpr int RPT = DK / 8;      // rows per thread
  const int64_t unit = blockIdx.x; // n * Hv + h
  const int n = (int)(unit / Hv), h = (int)(unit % Hv);
  const int hq = h / (Hv / Hqk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane >> 2, cg = lane & 3;
  const int col = warp * 16 + cg * 4;

  float* S = state + unit * (int64_t)(DK * DV);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(S + (rg + 8 * i) * DV + col);

  const __nv_bfloat16* kp = k + ((int64_t)n * Hqk + hq) * DK;
  const __nv_bfloat16* qp = q + ((int64_t)n * Hqk + hq) * DK;
  float kr[RPT], qr[RPT], ar[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    kr[i] = bf16_to_f32(kp[rg + 8 * i]);
    qr[i] = bf16_to_f32(qp[rg + 8 * i]);
  }
  if (KDA) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) ar[i] = expf(g[unit * DK + rg + 8 * i]);
  } else {
    const float a = expf(g[unit]);
#pragma unroll
    for (int i = 0; i < RPT; ++i) ar[i] = a;
  }
  const float b = beta[unit];
  const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(v + unit * DV + col);
  const float2 v01 = __bfloat1622float2(vp[0]);
  const float2 v23 = __bfloat1622float2(vp[1]);

  // S' = a S ; p = S'^T k (partial over my rows, then over the 8 row groups)
  float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    s[i].x *= ar[i]; s[i].y *= ar[i]; s[i].z *= ar[i]; s[i].w *= ar[i];
    p.x = fmaf(s[i].x, kr[i], p.x); p.y = fmaf(s[i].y, kr[i], p.y);
    p.z = fmaf(s[i].z, kr[i], p.z); p.w = fmaf(s[i].w, kr[i], p.w);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    p.x += __shfl_xor_sync(0xffffffffu, p.x, off); p.y += __shfl_xor_sync(0xffffffffu, p.y, off);
    p.z += __shfl_xor_sync(0xffffffffu, p.z, off); p.w += __shfl_xor_sync(0xffffffffu, p.w, off);
  }
  const float4 d = make_float4(b * (v01.x - p.x), b * (v01.y - p.y), b * (v23.x - p.z), b * (v23.y - p.w));

  // S = S' + k d^T ; o = S^T q
  float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    s[i].x = fmaf(kr[i], d.x, s[i].x); s[i].y = fmaf(kr[i], d.y, s[i].y);
    s[i].z = fmaf(kr[i], d.z, s[i].z); s[i].w = fmaf(kr[i], d.w, s[i].w);
    ov.x = fmaf(s[i].x, qr[i], ov.x); ov.y = fmaf(s[i].y, qr[i], ov.y);
    ov.z = fmaf(s[i].z, qr[i], ov.z); ov.w = fmaf(s[i].w, qr[i], ov.w);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(s[i].x), fabsf(s[i].y)), fmaxf(fabsf(s[i].z), fabsf(s[i].w))));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    ov.x += __shfl_xor_sync(0xffffffffu, ov.x, off); ov.y += __shfl_xor_sync(0xffffffffu, ov.y, off);
    ov.z += __shfl_xor_sync(0xffffffffu, ov.z, off); ov.w += __shfl_xor_sync(0xffffffffu, ov.w, off);
  }
  if (rg == 0)
    *reinterpret_cast<float4*>(o + unit * DV + col) =
        make_float4(scale * ov.x, scale * ov.y, scale * ov.z, scale * ov.w);

  if (state_qdq == 2) {
    // INT8 blocks: one key row x 32 value columns = one row of warps 2 b and 2 b + 1
    __shared__ float rmax[NW][DK];
    float m[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      m[i] = fmaxf(fmaxf(fabsf(s[i].x), fabsf(s[i].y)), fmaxf(fabsf(s[i].z), fabsf(s[i].w)));
      m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 1));
      m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 2));
      if (cg == 0) rmax[warp][rg + 8 * i] = m[i];
    }
    __syncthreads();
    // the 4 lanes of a row group share its rows: lane cg computes the scales of rows i = cg mod 4
    // and hands them to the other three
    float scl[RPT / 4], rcl[RPT / 4];
#pragma unroll
    for (int j = 0; j < RPT / 4; ++j) {
      const int i = 4 * j + cg;
      float bm = m[4 * j];
#pragma unroll
      for (int c = 1; c < 4; ++c) bm = c == cg ? m[4 * j + c] : bm;   // m[i] without dynamic indexing
      scl[j] = int8_scale(fmaxf(bm, rmax[warp ^ 1][rg + 8 * i]));
      rcl[j] = __frcp_rn(scl[j]);
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int src = (lane & ~3) | (i & 3);
      const float sc = __shfl_sync(0xffffffffu, scl[i >> 2], src), rc = __shfl_sync(0xffffffffu, rcl[i >> 2], src);
      s[i] = make_float4(int8_qdq_rcp(s[i].x, rc, sc), int8_qdq_rcp(s[i].y, rc, sc), int8_qdq_rcp(s[i].z, rc, sc),
                         int8_qdq_rcp(s[i].w, rc, sc));
    }
  } else if (state_qdq) {
    // one tile = all DK rows x 64 columns = 4 consecutive warps
    __shared__ float wmax[NW];
    amax = warp_max(amax);
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    const int t0 = (warp / 4) * 4;
    const float tmax = fmaxf(fmaxf(wmax[t0], wmax[t0 + 1]), fmaxf(wmax[t0 + 2], wmax[t0 + 3]));
    const float sc = qdq_scale(tmax), rc = __frcp_rn(sc);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const __nv_fp8x2_e4m3 c01(make_float2(__fmul_rn(s[i].x, rc), __fmul_rn(s[i].y, rc)));
      const __nv_fp8x2_e4m3 c23(make_float2(__fmul_rn(s[i].z, rc), __fmul_rn(s[i].w, rc)));
      const float2 f01 = static_cast<float2>(c01), f23 = static_cast<float2>(c23);
      s[i] = make_float4(__fmul_rn(f01.x, sc), __fmul_rn(f01.y, sc), __fmul_rn(f23.x, sc), __fmul_rn(f23.y, sc));
    }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(S + (rg + 8 * i) * DV + col) = s[i];
}

template <int DK, int DV, bool KDA>
cudaError_t launch_decode_t(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            float* state, float* o, int N, int Hqk, int Hv, float scale, int state_qdq,
                            cudaStream_t stream) {
  const int64_t units = (int64_t)N * Hv;
  if (units == 0) return cudaSuccess;
  decode_kernel<DK, DV, KDA><<<(unsigned)units, DV * 2, 0, stream>>>(
      (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, g, beta, state, o, Hqk, Hv,
      scale, state_qdq);
  return cudaGetLastError();
}

template <bool KDA>
cudaError_t dispatch_dv(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        float* state, float* o, int N, int Hqk, int Hv, int dk, int dv, float scale,
                        int state_qdq, cudaStream_t s) {
#define GDN_DEC(DKV, DVV)                                                                             \
  if (dk == DKV && dv == DVV)                                                                         \
    return launch_decode_t<DKV, DVV, KDA>(q, k, v, g, beta, state, o, N, Hqk, Hv, scale, state_qdq, s);
  GDN_DEC(64, 64) GDN_DEC(64, 128) GDN_DEC(64, 256) GDN_DEC(128, 64) GDN_DEC(128, 128) GDN_DEC(128, 256)
#undef GDN_DEC
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, float* o, int N, int Hqk, int Hv, int dk, int dv, float scale,
                          int state_qdq, int kda, cudaStream_t stream) {
  if (kda) return dispatch_dv<true>(q, k, v, g, beta, state, o, N, Hqk, Hv, dk, dv, scale, state_qdq, stream);
  return dispatch_dv<false>(q, k, v, g, beta, state, o, N, Hqk, Hv, dk, dv, scale, state_qdq, stream);
}

}  // namespace gdn
