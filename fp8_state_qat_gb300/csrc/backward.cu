// backward.cu -- gradients of the gated-delta-rule forward with straight-through state QDQ.
//
// What is differentiated ("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core
// QAT/QAD workflow" step 4: recurrent surrogate gradients with an identity straight-through
// estimator through QDQ; "GDN state/W QAT foundation": identity straight-through gradients): the
// token recurrence S_t = a_t S_{t-1} + b_t k_t (v_t - a_t S_{t-1}^T k_t)^T, o_t = scale S_t^T q_t
// (a_t = exp(g_t), KDA: row c scaled by exp(g_t[c])), with the state QDQ after every 64th token of
// a sequence in the forward values and the identity in the backward.
//
// Per token, with P the state before token t, P' = a o P, u = v - P'^T k, S = P' + b k u^T and dS
// the gradient reaching S (the o_t term scale q do^T added first):
//   dq = scale S do,  dv = du = b dS^T k,  db = k^T dS u,  dk = b dS u - P' du,
//   dP' = dS - k du^T,  dg = (dL/da) a = <dP', P> a = <dP', P'> (KDA: per key row),  dS_{t-1} = a o dP'.
// After the first token, dS is dh0.
//
// Apart from the state QDQ (a tile or block spans columns) and the quantities summed over the value
// columns (dq, dk, db, dg), the recurrence and its backward are column-local, so the work splits
// into one CTA per (sequence, head, 64-column value slab) -- the E4M3 tile width, so the forward
// QDQ stays CTA-local -- and a persistent grid walks those units, two CTAs per SM. Each CTA uses the
// decode kernel's thread layout (warp w owns slab columns [16 w, 16 w + 16); lane 4 rg + cg holds
// rows rg + 8 i and 4 columns): the first pass runs the forward recurrence, QDQ included, and
// stores the state entering every 64-token chunk; the second pass takes the chunks in reverse,
// recomputes the chunk's token states into the CTA's scratch, then walks its tokens backward with
// dS in registers. Column sums (over key rows) are warp shuffles; row sums (over the slab's
// columns) go through shared memory. The slab partials of dq, dk, db and dg land in the workspace
// and a second kernel sums them -- over slabs, and with GQA over the value heads that share a q/k
// head -- in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;
  const float* dout;    // [tokens, Hv, dv]
  const float* dhT;     // [N, Hv, dk, dv] or null
  float* part_q;        // [slabs][tokens, Hv, dk]: per-slab, per-v-head dq
  float* part_k;        // same for dk
  float* part_b;        // [slabs][tokens, Hv]: db
  float* part_g;        // [slabs][tokens, Hv] (KDA [slabs][tokens, Hv, dk]): dg
  float* grad_v;        // [tokens, Hv, dv]
  float* dh0;           // [N, Hv, dk, dv] or null
  float* ckpt;          // per (chunk slot, v-head): the state entering the chunk
  float* scratch;       // per CTA: the 64 slab states before the tokens of the current chunk
  int64_t tokens;
  int T, N, Hqk, Hv, dv;
  float scale;
  int state_qdq;
};

constexpr int SL = 64;        // value columns per CTA (one E4M3 tile)
constexpr int NW = SL / 16;   // warps per CTA

template <int DK>
struct BwdSmem {
  float rs[NW][DK][4];   // per warp, per key row: partial row sums
  float tot[NW][2];      // per warp partial full sums
  float wmax[NW];
  float rmax[NW][DK];
};

// ---- the forward step on the register state (decode layout) ----
template <int DK, bool KDA>
__device__ __forceinline__ void load_token(const BwdParams& p, int64_t tok, int h, int hq, int rg, int col,
                                           float* kr, float* qr, float* ar, float& b, float4& vv, float4& dov) {
  constexpr int RPT = DK / 8;
  const __nv_bfloat16* kp = p.k + (tok * p.Hqk + hq) * DK;
  const __nv_bfloat16* qp = p.q + (tok * p.Hqk + hq) * DK;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    kr[i] = bf16_to_f32(kp[rg + 8 * i]);
    qr[i] = bf16_to_f32(qp[rg + 8 * i]);
  }
  if (KDA) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) ar[i] = expf(p.g[(tok * p.Hv + h) * DK + rg + 8 * i]);
  } else {
    const float a = expf(p.g[tok * p.Hv + h]);
#pragma unroll
    for (int i = 0; i < RPT; ++i) ar[i] = a;
  }
  b = p.beta[tok * p.Hv + h];
  const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(p.v + (tok * p.Hv + h) * p.dv + col);
  const float2 v01 = __bfloat1622float2(vp[0]), v23 = __bfloat1622float2(vp[1]);
  vv = make_float4(v01.x, v01.y, v23.x, v23.y);
  dov = *reinterpret_cast<const float4*>(p.dout + (tok * p.Hv + h) * p.dv + col);
}

// column sums over the key rows of this warp's 4 columns per lane: partial over RPT rows, then the
// 8 row groups (lane bits 2..4)
__device__ __forceinline__ float4 col_sum(float4 x) {
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    x.x += __shfl_xor_sync(0xffffffffu, x.x, off); x.y += __shfl_xor_sync(0xffffffffu, x.y, off);
    x.z += __shfl_xor_sync(0xffffffffu, x.z, off); x.w += __shfl_xor_sync(0xffffffffu, x.w, off);
  }
  return x;
}

// S <- a S + b k (v - (a S)^T k)^T for one token (P' and u as in the header); returns u
template <int DK>
__device__ __forceinline__ void fwd_step(float4 (&s)[DK / 8], const float* kr, const float* ar, float b, float4 vv) {
  constexpr int RPT = DK / 8;
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    s[i].x *= ar[i]; s[i].y *= ar[i]; s[i].z *= ar[i]; s[i].w *= ar[i];
    pk.x = fmaf(s[i].x, kr[i], pk.x); pk.y = fmaf(s[i].y, kr[i], pk.y);
    pk.z = fmaf(s[i].z, kr[i], pk.z); pk.w = fmaf(s[i].w, kr[i], pk.w);
  }
  pk = col_sum(pk);
  const float4 d = make_float4(b * (vv.x - pk.x), b * (vv.y - pk.y), b * (vv.z - pk.z), b * (vv.w - pk.w));
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    s[i].x = fmaf(kr[i], d.x, s[i].x); s[i].y = fmaf(kr[i], d.y, s[i].y);
    s[i].z = fmaf(kr[i], d.z, s[i].z); s[i].w = fmaf(kr[i], d.w, s[i].w);
  }
}

// the forward's state QDQ on the register state (E4M3 tiles of 64 columns = 4 warps; INT8 blocks
// of one row x 32 columns = two warps); one barrier
template <int DK>
__device__ __forceinline__ void state_qdq(float4 (&s)[DK / 8], int codec, BwdSmem<DK>& sm, int warp, int lane,
                                          int rg, int cg) {
  constexpr int RPT = DK / 8;
  if (codec == 2) {
    float m[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      m[i] = fmaxf(fmaxf(fabsf(s[i].x), fabsf(s[i].y)), fmaxf(fabsf(s[i].z), fabsf(s[i].w)));
      m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 1));
      m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 2));
      if (cg == 0) sm.rmax[warp][rg + 8 * i] = m[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float sc = int8_scale(fmaxf(m[i], sm.rmax[warp ^ 1][rg + 8 * i])), rc = __frcp_rn(sc);
      s[i] = make_float4(int8_qdq_rcp(s[i].x, rc, sc), int8_qdq_rcp(s[i].y, rc, sc), int8_qdq_rcp(s[i].z, rc, sc),
                         int8_qdq_rcp(s[i].w, rc, sc));
    }
  } else {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(s[i].x), fabsf(s[i].y)), fmaxf(fabsf(s[i].z), fabsf(s[i].w))));
    amax = warp_max(amax);
    if (lane == 0) sm.wmax[warp] = amax;
    __syncthreads();
    const float tmax = fmaxf(fmaxf(sm.wmax[0], sm.wmax[1]), fmaxf(sm.wmax[2], sm.wmax[3]));   // the slab
    const float sc = qdq_scale(tmax), rc = __frcp_rn(sc);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const __nv_fp8x2_e4m3 c01(make_float2(__fmul_rn(s[i].x, rc), __fmul_rn(s[i].y, rc)));
      const __nv_fp8x2_e4m3 c23(make_float2(__fmul_rn(s[i].z, rc), __fmul_rn(s[i].w, rc)));
      const float2 f01 = static_cast<float2>(c01), f23 = static_cast<float2>(c23);
      s[i] = make_float4(__fmul_rn(f01.x, sc), __fmul_rn(f01.y, sc), __fmul_rn(f23.x, sc), __fmul_rn(f23.y, sc));
    }
  }
  __syncthreads();   // the next QDQ's shared-memory writes come after every thread's reads
}

template <int DK, bool KDA>
__global__ void __launch_bounds__(SL * 2, 2) chunk_bwd_kernel(const BwdParams p) {
  constexpr int RPT = DK / 8;
  __shared__ BwdSmem<DK> sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane >> 2, cg = lane & 3;
  const int nslab = p.dv / SL;
  const int64_t units = (int64_t)p.N * p.Hv * nslab;
  float* const scr = p.scratch + (int64_t)blockIdx.x * 64 * DK * SL;
  auto sat = [&](int r, int i) { return reinterpret_cast<float4*>(scr + ((int64_t)r * DK + rg + 8 * i) * SL + warp * 16 + cg * 4); };

  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int slab = (int)(unit % nslab);
    const int64_t nh = unit / nslab;   // n * Hv + h
    const int n = (int)(nh / p.Hv), h = (int)(nh % p.Hv);
    const int hq = h / (p.Hv / p.Hqk);
    const int col = slab * SL + warp * 16 + cg * 4;   // this lane's first value column
    const int64_t t0 = p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
    const int64_t len = p.cu ? (int64_t)p.cu[n + 1] - t0 : (int64_t)p.T;
    const int64_t nch = (len + 63) / 64;
    const int64_t slot0 = t0 / 64 + n;
    const int64_t st = (int64_t)DK * p.dv;   // one state
    auto srow = [&](const float* base, int i) { return base + (int64_t)(rg + 8 * i) * p.dv + col; };
    auto ck = [&](int64_t c) { return p.ckpt + ((slot0 + c) * p.Hv + h) * st; };
    float kr[RPT], qr[RPT], ar[RPT], b;
    float4 vv, dov;

    // ---- pass 1: the forward recurrence, storing the state entering every chunk ----
    float4 s[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      s[i] = p.h0 ? *reinterpret_cast<const float4*>(srow(p.h0 + nh * st, i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t t = 0; t < len; ++t) {
      if (t % 64 == 0) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(const_cast<float*>(srow(ck(t / 64), i))) = s[i];
      }
      load_token<DK, KDA>(p, t0 + t, h, hq, rg, col, kr, qr, ar, b, vv, dov);
      fwd_step<DK>(s, kr, ar, b, vv);
      if (p.state_qdq && (t + 1) % 64 == 0) state_qdq<DK>(s, p.state_qdq, sm, warp, lane, rg, cg);
    }

    // ---- pass 2: chunks in reverse; dS in registers ----
    float4 ds[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      ds[i] = p.dhT ? *reinterpret_cast<const float4*>(srow(p.dhT + nh * st, i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t c = nch - 1; c >= 0; --c) {
      const int L = (int)((len - c * 64) < 64 ? (len - c * 64) : 64);
      // the chunk's token states (before each token) into the scratch
#pragma unroll
      for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(srow(ck(c), i));
      for (int r = 0; r < L; ++r) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) *sat(r, i) = s[i];
        if (r + 1 < L) {
          load_token<DK, KDA>(p, t0 + c * 64 + r, h, hq, rg, col, kr, qr, ar, b, vv, dov);
          fwd_step<DK>(s, kr, ar, b, vv);
        }
      }
      for (int r = L - 1; r >= 0; --r) {
        const int64_t tok = t0 + c * 64 + r;
        load_token<DK, KDA>(p, tok, h, hq, rg, col, kr, qr, ar, b, vv, dov);
        float4 pp[RPT];   // P' = a o P
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float4 P = *sat(r, i);
          pp[i] = make_float4(ar[i] * P.x, ar[i] * P.y, ar[i] * P.z, ar[i] * P.w);
        }
        // u = v - P'^T k
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          u.x = fmaf(pp[i].x, kr[i], u.x); u.y = fmaf(pp[i].y, kr[i], u.y);
          u.z = fmaf(pp[i].z, kr[i], u.z); u.w = fmaf(pp[i].w, kr[i], u.w);
        }
        u = col_sum(u);
        u = make_float4(vv.x - u.x, vv.y - u.y, vv.z - u.z, vv.w - u.w);
        // dS += scale q do^T; du = b dS^T k
        const float4 sdo = make_float4(p.scale * dov.x, p.scale * dov.y, p.scale * dov.z, p.scale * dov.w);
        float4 du = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          ds[i].x = fmaf(qr[i], sdo.x, ds[i].x); ds[i].y = fmaf(qr[i], sdo.y, ds[i].y);
          ds[i].z = fmaf(qr[i], sdo.z, ds[i].z); ds[i].w = fmaf(qr[i], sdo.w, ds[i].w);
          du.x = fmaf(ds[i].x, kr[i], du.x); du.y = fmaf(ds[i].y, kr[i], du.y);
          du.z = fmaf(ds[i].z, kr[i], du.z); du.w = fmaf(ds[i].w, kr[i], du.w);
        }
        du = col_sum(du);
        du = make_float4(b * du.x, b * du.y, b * du.z, b * du.w);
        if (rg == 0) *reinterpret_cast<float4*>(p.grad_v + (tok * p.Hv + h) * p.dv + col) = du;
        // row sums over this lane's 4 columns: r0 = S do (S = P' + b k u^T), r1 = dS u, r2 = P' du,
        // r3 = dP' . P' with dP' = dS - k du^T
        float r0[RPT], r1[RPT], r2[RPT], r3[RPT];
        const float4 bu = make_float4(b * u.x, b * u.y, b * u.z, b * u.w);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float4 S = make_float4(fmaf(kr[i], bu.x, pp[i].x), fmaf(kr[i], bu.y, pp[i].y), fmaf(kr[i], bu.z, pp[i].z),
                                       fmaf(kr[i], bu.w, pp[i].w));
          r0[i] = S.x * dov.x + S.y * dov.y + S.z * dov.z + S.w * dov.w;
          r1[i] = ds[i].x * u.x + ds[i].y * u.y + ds[i].z * u.z + ds[i].w * u.w;
          r2[i] = pp[i].x * du.x + pp[i].y * du.y + pp[i].z * du.z + pp[i].w * du.w;
          const float4 dpp = make_float4(fmaf(-kr[i], du.x, ds[i].x), fmaf(-kr[i], du.y, ds[i].y),
                                         fmaf(-kr[i], du.z, ds[i].z), fmaf(-kr[i], du.w, ds[i].w));
          // dg = (dL/da) a = <dP', P> a = <dP', P'> (per key row for KDA)
          r3[i] = dpp.x * pp[i].x + dpp.y * pp[i].y + dpp.z * pp[i].z + dpp.w * pp[i].w;
          ds[i] = make_float4(ar[i] * dpp.x, ar[i] * dpp.y, ar[i] * dpp.z, ar[i] * dpp.w);   // dS_{t-1}
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
#pragma unroll
          for (int off = 1; off < 4; off <<= 1) {
            r0[i] += __shfl_xor_sync(0xffffffffu, r0[i], off);
            r1[i] += __shfl_xor_sync(0xffffffffu, r1[i], off);
            r2[i] += __shfl_xor_sync(0xffffffffu, r2[i], off);
            r3[i] += __shfl_xor_sync(0xffffffffu, r3[i], off);
          }
          if (cg == 0) {
            sm.rs[warp][rg + 8 * i][0] = r0[i];
            sm.rs[warp][rg + 8 * i][1] = r1[i];
            sm.rs[warp][rg + 8 * i][2] = r2[i];
            sm.rs[warp][rg + 8 * i][3] = r3[i];
          }
        }
        __syncthreads();
        // per key row cr (threads cr < DK): the slab's sums over its warps, in warp order
        const int64_t ph = (int64_t)slab * p.tokens * p.Hv + tok * p.Hv + h;   // slab partial index of (tok, h)
        float kb_c = 0.f, dg_c = 0.f;
        if (threadIdx.x < DK) {
          const int cr = threadIdx.x;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            a0 += sm.rs[w][cr][0]; a1 += sm.rs[w][cr][1]; a2 += sm.rs[w][cr][2]; a3 += sm.rs[w][cr][3];
          }
          const float kc = bf16_to_f32(p.k[(tok * p.Hqk + hq) * DK + cr]);
          p.part_q[ph * DK + cr] = p.scale * a0;
          p.part_k[ph * DK + cr] = b * a1 - a2;
          kb_c = kc * a1;   // contribution to db
          dg_c = a3;        // contribution to dg (GDN: summed over the rows)
          if (KDA) p.part_g[ph * DK + cr] = a3;
        }
        // db and (GDN) dg: sums over the key rows (warps 0 .. DK/32 - 1 hold them)
        if (warp < DK / 32) {
          float x0 = kb_c, x1 = dg_c;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            x0 += __shfl_xor_sync(0xffffffffu, x0, off);
            x1 += __shfl_xor_sync(0xffffffffu, x1, off);
          }
          if (lane == 0) {
            sm.tot[warp][0] = x0;
            sm.tot[warp][1] = x1;
          }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          float db = 0.f, dg = 0.f;
#pragma unroll
          for (int w = 0; w < DK / 32; ++w) {
            db += sm.tot[w][0];
            dg += sm.tot[w][1];
          }
          p.part_b[ph] = db;
          if (!KDA) p.part_g[ph] = dg;
        }
        __syncthreads();   // sm.rs / sm.tot are rewritten by the next token
      }
    }
    if (p.dh0) {
#pragma unroll
      for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(p.dh0 + nh * st + (int64_t)(rg + 8 * i) * p.dv + col) = ds[i];
    }
  }
}

// out[e] = sum over slabs s < nslab and value heads j < G of part[s * slab_stride + src(e, j)],
// src(e, j) = ((e / inner) G + j) inner + e mod inner (dq / dk: inner = dk, G value heads per q/k
// head; db, dg: G = 1), in that fixed order
__global__ void sum_parts_kernel(const float* __restrict__ part, float* __restrict__ out, int64_t n_out, int nslab,
                                 int64_t slab_stride, int G, int inner) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_out; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t base = (e / inner) * G * inner + e % inner;
    float acc = 0.f;
    for (int s = 0; s < nslab; ++s)
      for (int j = 0; j < G; ++j) acc += part[s * slab_stride + base + (int64_t)j * inner];
    out[e] = acc;
  }
}

constexpr int kBwdCtas = 2 * 152;   // two CTAs per GB300 SM at most; each owns a 64-state scratch

template <int DK, bool KDA>
cudaError_t launch_t(const BwdParams& bp, int64_t units, cudaStream_t stream) {
  int dev = 0, sms = kBwdCtas / 2;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaGetLastError();
  int64_t grid = units < 2 * (int64_t)sms ? units : 2 * (int64_t)sms;
  if (grid > kBwdCtas) grid = kBwdCtas;
  chunk_bwd_kernel<DK, KDA><<<(unsigned)grid, SL * 2, 0, stream>>>(bp);
  return cudaGetLastError();
}

cudaError_t sum_parts(const float* part, float* out, int64_t n_out, int nslab, int64_t slab_stride, int G, int inner,
                      cudaStream_t stream) {
  if (n_out == 0) return cudaSuccess;
  const int64_t blocks = (n_out + 255) / 256 < 152 * 32 ? (n_out + 255) / 256 : 152 * 32;
  sum_parts_kernel<<<(unsigned)blocks, 256, 0, stream>>>(part, out, n_out, nslab, slab_stride, G, inner);
  return cudaGetLastError();
}

}  // namespace

BwdLayout chunk_bwd_layout(const ChunkProblem& p) {
  BwdLayout l{};
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const int64_t tokens = (int64_t)p.B * p.T;
  const int64_t slots = tokens / 64 + p.N;
  const int nslab = p.dv / SL;
  const int64_t units = (int64_t)p.N * p.Hv * nslab;
  const int64_t ctas = units < kBwdCtas ? units : kBwdCtas;
  const size_t part = (size_t)nslab * tokens * p.Hv * 4;
  l.off_ckpt = up(kStatusBytes);
  l.off_scratch = up(l.off_ckpt + (size_t)slots * p.Hv * p.dk * p.dv * 4);
  l.off_part_q = up(l.off_scratch + (size_t)ctas * 64 * p.dk * SL * 4);
  l.off_part_k = up(l.off_part_q + part * p.dk);
  l.off_part_b = up(l.off_part_k + part * p.dk);
  l.off_part_g = up(l.off_part_b + part);
  l.total = up(l.off_part_g + part * (p.kda ? p.dk : 1));
  return l;
}

cudaError_t launch_chunk_bwd(const ChunkProblem& p, const BwdGrads& gr, void* ws, cudaStream_t stream) {
  const BwdLayout lay = chunk_bwd_layout(p);
  const int nslab = p.dv / SL;
  const int64_t units = (int64_t)p.N * p.Hv * nslab;
  if (units == 0) return cudaSuccess;
  unsigned char* w = static_cast<unsigned char*>(ws);
  const int64_t tokens = (int64_t)p.B * p.T;
  float* pq = reinterpret_cast<float*>(w + lay.off_part_q);
  float* pk = reinterpret_cast<float*>(w + lay.off_part_k);
  float* pb = reinterpret_cast<float*>(w + lay.off_part_b);
  float* pg = reinterpret_cast<float*>(w + lay.off_part_g);
  BwdParams bp{(const __nv_bfloat16*)p.q, (const __nv_bfloat16*)p.k, (const __nv_bfloat16*)p.v, p.g, p.beta, p.h0,
               p.cu, gr.dout, gr.dhT, pq, pk, pb, pg, gr.dv, gr.dh0,
               reinterpret_cast<float*>(w + lay.off_ckpt), reinterpret_cast<float*>(w + lay.off_scratch), tokens,
               p.T, p.N, p.Hqk, p.Hv, p.dv, p.scale, p.state_qdq};
  cudaError_t e = cudaErrorInvalidValue;
  if (p.dk == 64) e = p.kda ? launch_t<64, true>(bp, units, stream) : launch_t<64, false>(bp, units, stream);
  if (p.dk == 128) e = p.kda ? launch_t<128, true>(bp, units, stream) : launch_t<128, false>(bp, units, stream);
  if (e != cudaSuccess || tokens == 0) return e;
  const int G = p.Hv / p.Hqk;
  const int64_t sh = tokens * p.Hv;   // per-slab stride in (token, v-head) units
  if ((e = sum_parts(pq, gr.dq, tokens * p.Hqk * p.dk, nslab, sh * p.dk, G, p.dk, stream)) != cudaSuccess) return e;
  if ((e = sum_parts(pk, gr.dk, tokens * p.Hqk * p.dk, nslab, sh * p.dk, G, p.dk, stream)) != cudaSuccess) return e;
  if ((e = sum_parts(pb, gr.dbeta, sh, nslab, sh, 1, 1, stream)) != cudaSuccess) return e;
  const int gk = p.kda ? p.dk : 1;
  return sum_parts(pg, gr.dg, sh * gk, nslab, sh * gk, 1, 1, stream);
}

}  // namespace gdn
