// handoff.cu -- the decode part of a prefill -> decode handoff.
//
// Schedule ("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD
// workflow", steps 2-3, and its "Ordinary state-QDQ path" flowchart): the first P_n tokens of
// sequence n run as chunked prefill that leaves a state without internal state QDQ (the chunk
// kernels, run with per-sequence lengths P_n); when tokens remain, the state is QDQ'd at the
// handoff and every remaining token is a decode step on the sequence's own tokens (teacher
// forced): read the state, S' = a S (KDA: row c scaled by a[c]), d = b (v - S'^T k),
// S = S' + k d^T, o = scale S^T q from the updated state, then QDQ (E4M3: all dk rows x 64 value
// columns per tile, scale amax / 448, 1 for an all-zero tile; INT8: one key row x 32 value columns per
// block, amax / 127) before the state is stored for the next token.
//
// One CTA per (sequence, head) keeps the state in registers across all of the sequence's
// decode tokens, so HBM sees the state once in and once out plus each token's q, k, v, g, beta
// and o. The thread layout and reduction order are the decode kernel's (so a decode token gives
// the same bits here and there): warp w owns value columns [16 w, 16 w + 16); lane = 4 rg + cg
// holds rows rg, rg + 8, ... and the 4 columns 16 w + 4 cg .. + 3; both dk-reductions are
// 3-level xor shuffles over lane bits 2..4 in a fixed order. The inputs of
// the next kAhead - 1 tokens are in flight (cp.async into a ring of shared-memory buffers)
// while a token is computed; the per-tile maxima alternate between two shared-memory slots.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

// One token's inputs, staged in shared memory by cp.async one token ahead.
template <int DK, int DV, bool KDA>
struct __align__(16) TokenBuf {
  __nv_bfloat16 k[DK], q[DK], v[DV];
  float g[KDA ? DK : 1];
  float b;
};

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Decode tokens whose inputs are in flight ahead of the one being computed: a token's
// arithmetic is a few hundred cycles, an HBM round trip about a microsecond.
constexpr int kAhead = 8;

// Issue the copies of token tok's inputs into buf (k, q, v in 16-byte pieces; g, beta in 4-byte
// pieces, so g needs only 4-byte alignment).
template <int DK, int DV, bool KDA>
__device__ __forceinline__ void stage_token(TokenBuf<DK, DV, KDA>& buf, const __nv_bfloat16* __restrict__ q,
                                            const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                                            const float* __restrict__ g, const float* __restrict__ beta, int64_t tok,
                                            int Hqk, int Hv, int h, int hq) {
  constexpr int NK = DK / 8, NV = DV / 8;   // 16-byte pieces of k (and q), of v
  const int tid = threadIdx.x;
  if (tid < NK) cp16(&buf.k[8 * tid], k + (tok * Hqk + hq) * DK + 8 * tid);
  else if (tid < 2 * NK) cp16(&buf.q[8 * (tid - NK)], q + (tok * Hqk + hq) * DK + 8 * (tid - NK));
  else if (tid < 2 * NK + NV) cp16(&buf.v[8 * (tid - 2 * NK)], v + (tok * Hv + h) * DV + 8 * (tid - 2 * NK));
  if (KDA) {
    if (tid < DK) cp4(&buf.g[tid], g + (tok * Hv + h) * DK + tid);
  } else if (tid == 0) {
    cp4(&buf.g[0], g + tok * Hv + h);
  }
  if (tid == 1) cp4(&buf.b, beta + tok * Hv + h);
}

// QDQ of the state registers: one tile = all DK rows x 64 columns = 4 consecutive warps. The
// state registers are column pairs (col, col + 1) and (col + 2, col + 3) so that the
// elementwise work runs as paired fp32 operations (fma / mul .f32x2, each lane rounded like
// its scalar form). EXACT: x / s as the correctly rounded quotient (the once-per-sequence QDQ at
// the handoff, bit for bit the fp32 definition); otherwise x times the rounded reciprocal of s
// (every decode token's QDQ; differs from the IEEE quotient's E4M3 code for ~2 in 10^7 elements).
template <int DK, int DV, bool EXACT = false>
__device__ __forceinline__ float qdq_state_regs(float2 (&sa)[DK / 8], float2 (&sb)[DK / 8], float amax, float* wmax,
                                                int warp, int lane) {
  constexpr int RPT = DK / 8;
  amax = warp_max(amax);
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  const int t0 = (warp / 4) * 4;
  const float tmax = fmaxf(fmaxf(wmax[t0], wmax[t0 + 1]), fmaxf(wmax[t0 + 2], wmax[t0 + 3]));
  const float sc = qdq_scale(tmax), rc = __frcp_rn(sc);
  const float2 sc2 = make_float2(sc, sc), rc2 = make_float2(rc, rc), nsc2 = make_float2(-sc, -sc);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    // a subnormal scale has no finite reciprocal: the IEEE divide then (tmax below ~3e-36)
    const float2 ya = !EXACT ? __fmul2_rn(sa[i], rc2)
                             : (sc >= 1.17549435e-38f ? quotient2(sa[i], nsc2, rc2)
                                                      : make_float2(__fdiv_rn(sa[i].x, sc), __fdiv_rn(sa[i].y, sc)));
    const float2 yb = !EXACT ? __fmul2_rn(sb[i], rc2)
                             : (sc >= 1.17549435e-38f ? quotient2(sb[i], nsc2, rc2)
                                                      : make_float2(__fdiv_rn(sb[i].x, sc), __fdiv_rn(sb[i].y, sc)));
    const __nv_fp8x2_e4m3 ca(ya), cb(yb);
    sa[i] = __fmul2_rn(static_cast<float2>(ca), sc2);
    sb[i] = __fmul2_rn(static_cast<float2>(cb), sc2);
  }
  return sc;
}

// INT8 block QDQ of the state registers (state_qdq == 2): one block = one key row x 32 value
// columns = that row's 8 lanes (cg 0..3) in warps 2 b and 2 b + 1. rmax: shared [NW][DK]. The
// caller keeps a barrier between one call's reads of rmax and the next call's writes.
template <int DK, int DV>
__device__ __forceinline__ void int8_state_regs(float2 (&sa)[DK / 8], float2 (&sb)[DK / 8], float (*rmax)[DK],
                                                int warp, int rg, int cg, float* srow) {
  constexpr int RPT = DK / 8;
  float m[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    m[i] = fmaxf(fmaxf(fabsf(sa[i].x), fabsf(sa[i].y)), fmaxf(fabsf(sb[i].x), fabsf(sb[i].y)));
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
    float bm = m[4 * j];
#pragma unroll
    for (int c = 1; c < 4; ++c) bm = c == cg ? m[4 * j + c] : bm;   // m[4 j + cg] without dynamic indexing
    scl[j] = int8_scale(fmaxf(bm, rmax[warp ^ 1][rg + 8 * (4 * j + cg)]));
    rcl[j] = __frcp_rn(scl[j]);
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int src = (lane & ~3) | (i & 3);
    const float sc = __shfl_sync(0xffffffffu, scl[i >> 2], src), rc = __shfl_sync(0xffffffffu, rcl[i >> 2], src);
    if (srow) srow[(rg + 8 * i) * (DV / kInt8BlockCols)] = sc;   // the final state's scales
    sa[i] = make_float2(int8_qdq_rcp(sa[i].x, rc, sc), int8_qdq_rcp(sa[i].y, rc, sc));
    sb[i] = make_float2(int8_qdq_rcp(sb[i].x, rc, sc), int8_qdq_rcp(sb[i].y, rc, sc));
  }
}

template <int DK, int DV, bool KDA>
__global__ void __launch_bounds__(DV * 2, (DV <= 128 ? 2 : 1))
handoff_suffix_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                      const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
                      const float* __restrict__ beta, const int32_t* __restrict__ cu,
                      const int32_t* __restrict__ plens, float* __restrict__ state, float* __restrict__ o, int T,
                      int Hqk, int Hv, float scale, int state_qdq, float* __restrict__ sscale) {
  constexpr int NW = DV / 16;
  constexpr int RPT = DK / 8;
  __shared__ float wmax[2][NW];
  __shared__ float rmax[NW][DK];   // INT8 codec: per-row maxima of each warp's 16 columns
  __shared__ __align__(16) TokenBuf<DK, DV, KDA> tb[kAhead];
  const int64_t unit = blockIdx.x;   // n * Hv + h
  const int n = (int)(unit / Hv), h = (int)(unit % Hv);
  const int hq = h / (Hv / Hqk);
  const int64_t t0 = cu ? (int64_t)cu[n] : (int64_t)n * T;
  const int64_t len = cu ? (int64_t)cu[n + 1] - t0 : (int64_t)T;
  const int64_t P = plens[n];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane >> 2, cg = lane & 3;
  const int col = warp * 16 + cg * 4;
  // final-state scales (layout: ChunkProblem::state_scales): E4M3 by lane 0 of each tile's first
  // warp; INT8 by the cg = 0 lanes of each block's first warp (rows rg + 8 i), inside the last QDQ
  float* const i8dst = (sscale && state_qdq == 2 && cg == 0 && (warp & 1) == 0)
                           ? sscale + unit * DK * (DV / kInt8BlockCols) + warp / 2
                           : nullptr;
  float last_tile = 0.f;
  if (P >= len) {   // no decode tokens: the prefill state stays as it is, not QDQ'd
    if (i8dst) {
#pragma unroll
      for (int i = 0; i < RPT; ++i) i8dst[(rg + 8 * i) * (DV / kInt8BlockCols)] = 0.f;
    } else if (sscale && state_qdq != 2 && lane == 0 && (warp & 3) == 0) {
      sscale[unit * (DV / 64) + warp / 4] = 0.f;
    }
    return;
  }

  float* S = state + unit * (int64_t)(DK * DV);
  float2 sa[RPT], sb[RPT];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float4 f = *reinterpret_cast<const float4*>(S + (rg + 8 * i) * DV + col);
    sa[i] = make_float2(f.x, f.y);
    sb[i] = make_float2(f.z, f.w);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  // tokens P .. P + kAhead - 2 in flight, one cp.async group each (empty groups past the end)
#pragma unroll 1
  for (int j = 0; j < kAhead - 1; ++j) {
    if (P + j < len) stage_token<DK, DV, KDA>(tb[j], q, k, v, g, beta, t0 + P + j, Hqk, Hv, h, hq);
    cp_commit();
  }
  int slot = 0;   // the per-tile maxima alternate between two slots, one barrier per QDQ
  if (state_qdq == 2) {
    int8_state_regs<DK, DV>(sa, sb, rmax, warp, rg, cg, nullptr);   // the handoff (decode tokens follow)
  } else if (state_qdq) {
    last_tile = qdq_state_regs<DK, DV, true>(sa, sb, amax, wmax[slot], warp, lane);   // the handoff
    slot ^= 1;
  }

  for (int64_t t = P; t < len; ++t) {
    const int i = (int)(t - P);
    cp_wait<kAhead - 2>();   // this thread's copies of token t have landed
    __syncthreads();         // ... and everyone's; every thread is done with token t - 1's buffer
    // token t + kAhead - 1 goes into the buffer token t - 1 used
    if (t + kAhead - 1 < len)
      stage_token<DK, DV, KDA>(tb[(i + kAhead - 1) % kAhead], q, k, v, g, beta, t0 + t + kAhead - 1, Hqk, Hv, h, hq);
    cp_commit();
    const TokenBuf<DK, DV, KDA>& in = tb[i % kAhead];
    float kr[RPT], qr[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      kr[i] = bf16_to_f32(in.k[rg + 8 * i]);
      qr[i] = bf16_to_f32(in.q[rg + 8 * i]);
    }
    const float a0 = KDA ? 0.f : expf(in.g[0]);
    const float b = in.b;
    const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(&in.v[col]);
    const float2 v01 = __bfloat1622float2(vp[0]), v23 = __bfloat1622float2(vp[1]);
    // S' = a S ; p = S'^T k
    float2 pa = make_float2(0.f, 0.f), pb = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float a = KDA ? expf(in.g[rg + 8 * i]) : a0;
      const float2 a2 = make_float2(a, a), k2 = make_float2(kr[i], kr[i]);
      sa[i] = __fmul2_rn(sa[i], a2);
      sb[i] = __fmul2_rn(sb[i], a2);
      pa = __ffma2_rn(sa[i], k2, pa);
      pb = __ffma2_rn(sb[i], k2, pb);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      pa.x += __shfl_xor_sync(0xffffffffu, pa.x, off); pa.y += __shfl_xor_sync(0xffffffffu, pa.y, off);
      pb.x += __shfl_xor_sync(0xffffffffu, pb.x, off); pb.y += __shfl_xor_sync(0xffffffffu, pb.y, off);
    }
    const float2 da = make_float2(b * (v01.x - pa.x), b * (v01.y - pa.y));
    const float2 db = make_float2(b * (v23.x - pb.x), b * (v23.y - pb.y));
    // S = S' + k d^T ; o = S^T q
    float2 oa = make_float2(0.f, 0.f), ob = make_float2(0.f, 0.f);
    amax = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float2 k2 = make_float2(kr[i], kr[i]), q2 = make_float2(qr[i], qr[i]);
      sa[i] = __ffma2_rn(k2, da, sa[i]);
      sb[i] = __ffma2_rn(k2, db, sb[i]);
      oa = __ffma2_rn(sa[i], q2, oa);
      ob = __ffma2_rn(sb[i], q2, ob);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(sa[i].x), fabsf(sa[i].y)), fmaxf(fabsf(sb[i].x), fabsf(sb[i].y))));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      oa.x += __shfl_xor_sync(0xffffffffu, oa.x, off); oa.y += __shfl_xor_sync(0xffffffffu, oa.y, off);
      ob.x += __shfl_xor_sync(0xffffffffu, ob.x, off); ob.y += __shfl_xor_sync(0xffffffffu, ob.y, off);
    }
    if (rg == 0)
      *reinterpret_cast<float4*>(o + ((t0 + t) * Hv + h) * DV + col) =
          make_float4(scale * oa.x, scale * oa.y, scale * ob.x, scale * ob.y);
    if (state_qdq == 2) {
      int8_state_regs<DK, DV>(sa, sb, rmax, warp, rg, cg, t + 1 == len ? i8dst : nullptr);
    } else if (state_qdq) {
      last_tile = qdq_state_regs<DK, DV>(sa, sb, amax, wmax[slot], warp, lane);
      slot ^= 1;
    }
  }
  cp_wait<0>();   // nothing may still be landing in shared memory when the CTA exits
  if (sscale && state_qdq != 2 && lane == 0 && (warp & 3) == 0) sscale[unit * (DV / 64) + warp / 4] = last_tile;
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    *reinterpret_cast<float4*>(S + (rg + 8 * i) * DV + col) = make_float4(sa[i].x, sa[i].y, sb[i].x, sb[i].y);
}

template <int DK, int DV, bool KDA>
cudaError_t launch_t(const ChunkProblem& p, const int32_t* plens, cudaStream_t stream) {
  const int64_t units = (int64_t)p.N * p.Hv;
  if (units == 0) return cudaSuccess;
  handoff_suffix_kernel<DK, DV, KDA><<<(unsigned)units, DV * 2, 0, stream>>>(
      (const __nv_bfloat16*)p.q, (const __nv_bfloat16*)p.k, (const __nv_bfloat16*)p.v, p.g, p.beta, p.cu, plens, p.hT,
      p.o, p.T, p.Hqk, p.Hv, p.scale, p.state_qdq, p.state_scales);
  return cudaGetLastError();
}

template <bool KDA>
cudaError_t dispatch(const ChunkProblem& p, const int32_t* plens, cudaStream_t s) {
#define GDN_HO(DKV, DVV) \
  if (p.dk == DKV && p.dv == DVV) return launch_t<DKV, DVV, KDA>(p, plens, s);
  GDN_HO(64, 64) GDN_HO(64, 128) GDN_HO(64, 256) GDN_HO(128, 64) GDN_HO(128, 128) GDN_HO(128, 256)
#undef GDN_HO
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_handoff_suffix(const ChunkProblem& p, const int32_t* plens, cudaStream_t stream) {
  if (!p.hT) return cudaErrorInvalidValue;
  return p.kda ? dispatch<true>(p, plens, stream) : dispatch<false>(p, plens, stream);
}

}  // namespace gdn
