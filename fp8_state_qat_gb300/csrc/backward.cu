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
// QDQ stays CTA-local -- and a persistent grid (one CTA per SM) walks those units. 256 threads:
// warp w owns slab columns [8 w, 8 w + 8); lane 4 rg + cg holds the dk / 8 consecutive key rows
// from (dk / 8) rg and the two columns 8 w + 2 cg, + 1, so a column sum over the key rows is a
// 3-level xor shuffle. The registers pair two adjacent key rows of one column, so k, q and a
// arrive as natural pairs for the paired fp32 instructions (fma / mul .f32x2) and only the
// per-column scalars of a token are broadcast.
//
// Pass 1 runs the forward recurrence, QDQ included, and stores the state entering every 64-token
// chunk. Pass 2 takes the chunks in reverse: the chunk's token inputs are staged in shared memory
// (cp.async), a forward sweep stores the state entering every 4-token sub-chunk in a per-CTA
// scratch small enough to stay in L2, and then each sub-chunk, last first, is recomputed from its
// checkpoint -- three states into per-thread shared-memory slots, the fourth left in registers --
// and walked backward with dS in registers. Per token one barrier: the row sums (over the slab's
// columns) are reduced within a lane quad by a reduce-scatter, then over the warps through a
// double-buffered shared array. The slab (and per-warp) partials of dq, dk, db and dg land in the
// workspace and a second kernel sums them -- over slabs, and with GQA over the value heads that
// share a q/k head -- in a fixed order.
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
  float* part_b;        // [slabs * dk / 32][tokens, Hv]: db per slab and reducing warp
  float* part_g;        // GDN: as part_b; KDA [slabs][tokens, Hv, dk]: dg
  float* grad_v;        // [tokens, Hv, dv]
  float* dh0;           // [N, Hv, dk, dv] or null
  float* ckpt;          // per (chunk slot, v-head): the state entering the chunk
  float* scratch;       // per CTA: the 16 sub-chunk checkpoints of the current chunk (thread-major)
  int64_t tokens;
  int T, N, Hqk, Hv, dv;
  float scale;
  int state_qdq;
};

constexpr int SL = 64;          // value columns per CTA (one E4M3 tile)
constexpr int NT = 256;         // threads per CTA
constexpr int NW = NT / 32;     // warps; warp w owns slab columns [8 w, 8 w + 8)
constexpr int SUB = 4;          // tokens per sub-chunk
constexpr int NSUB = kChunk / SUB;

// One token's inputs in shared memory (byte offsets): k, q (dk bf16 each), the slab's v (bf16) and
// dout (fp32) columns, the gate(s) (fp32, turned into a = exp(g) after staging), beta.
template <int DK, bool KDA>
struct Rec {
  static constexpr int K = 0, Q = 2 * DK, V = 4 * DK, DO = 4 * DK + 2 * SL, G = 4 * DK + 6 * SL;
  static constexpr int NG = KDA ? DK : 1;
  static constexpr int B = G + 4 * NG;
  static constexpr int BYTES = (B + 4 + 15) / 16 * 16;
  static constexpr int N16 = DK / 4 + SL / 8 + SL / 4 + (KDA ? DK / 4 : 0);   // 16-byte pieces
  static constexpr int NP = N16 + (KDA ? 1 : 2);                               // + 4-byte g (GDN), beta
};

template <int DK, bool KDA>
struct BwdSmem {
  alignas(16) unsigned char stage[kChunk * Rec<DK, KDA>::BYTES];
  float2 slot[SUB - 1][DK / 8][NT];   // per-thread copies of the sub-chunk's first token states
                                      // (the row sums below are indexed by rs_slot of the key row)
  float4 rs[2][NW][DK];               // per token (double-buffered), warp, key row: 4 row sums
  float wmax[NW];
  float rmax[NW][DK];
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

// Stage tokens tok0 .. tok0 + count - 1 (count <= 64) of head (h, hq), value slab `slab`, into
// consecutive records at dst; every thread issues its share of the pieces (no commit here).
template <int DK, bool KDA>
__device__ __forceinline__ void stage_tokens(const BwdParams& p, unsigned char* dst, int64_t tok0, int count, int h,
                                             int hq, int slab) {
  using R = Rec<DK, KDA>;
  for (int e = threadIdx.x; e < count * R::NP; e += NT) {
    const int r = e / R::NP;
    int j = e - r * R::NP;
    const int64_t tok = tok0 + r, th = tok * p.Hv + h;
    unsigned char* d = dst + r * R::BYTES;
    if (j < DK / 8) { cp16(d + R::K + 16 * j, p.k + (tok * p.Hqk + hq) * DK + 8 * j); continue; }
    j -= DK / 8;
    if (j < DK / 8) { cp16(d + R::Q + 16 * j, p.q + (tok * p.Hqk + hq) * DK + 8 * j); continue; }
    j -= DK / 8;
    if (j < SL / 8) { cp16(d + R::V + 16 * j, p.v + th * p.dv + slab * SL + 8 * j); continue; }
    j -= SL / 8;
    if (j < SL / 4) { cp16(d + R::DO + 16 * j, p.dout + th * p.dv + slab * SL + 4 * j); continue; }
    j -= SL / 4;
    if (KDA) {
      if (j < DK / 4) { cp16(d + R::G + 16 * j, p.g + th * DK + 4 * j); continue; }
      j -= DK / 4;
    } else {
      if (j == 0) { cp4(d + R::G, p.g + th); continue; }
      j -= 1;
    }
    cp4(d + R::B, p.beta + th);
  }
}

// g -> a = exp(g) in `count` staged records (after the copies are visible to every thread)
template <int DK, bool KDA>
__device__ __forceinline__ void exp_gates(unsigned char* rec0, int count) {
  using R = Rec<DK, KDA>;
  for (int e = threadIdx.x; e < count * R::NG; e += NT) {
    const int r = e / R::NG;
    float* gp = reinterpret_cast<float*>(rec0 + r * R::BYTES + R::G) + (e - r * R::NG);
    *gp = expf(*gp);
  }
}

// This thread's view of one staged token: k, q and a on its key rows as (row 2 j, row 2 j + 1)
// pairs; beta; v and dout on its two columns.
template <int DK>
struct TokView {
  float2 k2[DK / 16], q2[DK / 16], a2[DK / 16];
  float b;
  float2 vv, dov;
};

template <int DK, bool KDA>
__device__ __forceinline__ void read_token(const unsigned char* rec, int rg, int c0, bool need_q, TokView<DK>& t) {
  using R = Rec<DK, KDA>;
  constexpr int RPT = DK / 8, NPR = RPT / 2;
  const uint4* kk = reinterpret_cast<const uint4*>(rec + R::K + 2 * RPT * rg);
  const uint4* qq = reinterpret_cast<const uint4*>(rec + R::Q + 2 * RPT * rg);
#pragma unroll
  for (int j = 0; j < RPT / 8; ++j) {
    const uint4 x = kk[j];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) t.k2[4 * j + e] = __bfloat1622float2(h[e]);
    if (need_q) {
      const uint4 y = qq[j];
      const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
      for (int e = 0; e < 4; ++e) t.q2[4 * j + e] = __bfloat1622float2(hq[e]);
    }
  }
  if (KDA) {
    const float4* ga = reinterpret_cast<const float4*>(rec + R::G + 4 * RPT * rg);
#pragma unroll
    for (int j = 0; j < RPT / 4; ++j) {
      const float4 x = ga[j];
      t.a2[2 * j] = make_float2(x.x, x.y);
      t.a2[2 * j + 1] = make_float2(x.z, x.w);
    }
  } else {
    const float a = *reinterpret_cast<const float*>(rec + R::G);
#pragma unroll
    for (int j = 0; j < NPR; ++j) t.a2[j] = make_float2(a, a);
  }
  t.b = *reinterpret_cast<const float*>(rec + R::B);
  t.vv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(rec + R::V + 2 * c0));
  t.dov = *reinterpret_cast<const float2*>(rec + R::DO + 4 * c0);
}

// column sums over the key rows: the two row halves of each pair, then the 8 row groups (lane bits 2..4)
__device__ __forceinline__ float2 col_sum(float2 acc0, float2 acc1) {
  float2 x = make_float2(acc0.x + acc0.y, acc1.x + acc1.y);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    x.x += __shfl_xor_sync(0xffffffffu, x.x, off);
    x.y += __shfl_xor_sync(0xffffffffu, x.y, off);
  }
  return x;
}

__device__ __forceinline__ float2 bcast(float x) { return make_float2(x, x); }

// a [dk, dv] state in global memory <-> this thread's pairs (s[c][j] = rows 2 j, 2 j + 1 of column c)
template <int DK>
__device__ __forceinline__ void load_state(float2 (&s)[2][DK / 16], const float* base, int64_t dv, int r0, int col) {
#pragma unroll
  for (int j = 0; j < DK / 16; ++j) {
    const float2 x = *reinterpret_cast<const float2*>(base + (int64_t)(r0 + 2 * j) * dv + col);
    const float2 y = *reinterpret_cast<const float2*>(base + (int64_t)(r0 + 2 * j + 1) * dv + col);
    s[0][j] = make_float2(x.x, y.x);
    s[1][j] = make_float2(x.y, y.y);
  }
}
template <int DK>
__device__ __forceinline__ void store_state(const float2 (&s)[2][DK / 16], float* base, int64_t dv, int r0, int col) {
#pragma unroll
  for (int j = 0; j < DK / 16; ++j) {
    *reinterpret_cast<float2*>(base + (int64_t)(r0 + 2 * j) * dv + col) = make_float2(s[0][j].x, s[1][j].x);
    *reinterpret_cast<float2*>(base + (int64_t)(r0 + 2 * j + 1) * dv + col) = make_float2(s[0][j].y, s[1][j].y);
  }
}

// S <- a S + b k (v - (a S)^T k)^T for one token
template <int DK>
__device__ __forceinline__ void fwd_step(float2 (&s)[2][DK / 16], const TokView<DK>& t) {
  constexpr int NPR = DK / 16;
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < NPR; ++j) {
    s[0][j] = __fmul2_rn(s[0][j], t.a2[j]);
    s[1][j] = __fmul2_rn(s[1][j], t.a2[j]);
    acc0 = __ffma2_rn(s[0][j], t.k2[j], acc0);
    acc1 = __ffma2_rn(s[1][j], t.k2[j], acc1);
  }
  const float2 pk = col_sum(acc0, acc1);
  const float2 d0 = bcast(t.b * (t.vv.x - pk.x)), d1 = bcast(t.b * (t.vv.y - pk.y));
#pragma unroll
  for (int j = 0; j < NPR; ++j) {
    s[0][j] = __ffma2_rn(t.k2[j], d0, s[0][j]);
    s[1][j] = __ffma2_rn(t.k2[j], d1, s[1][j]);
  }
}

// the forward's state QDQ on the register state (E4M3: the slab is one tile, all 8 warps; INT8: a
// block is one key row of 32 columns = warps 4 b .. 4 b + 3); barriers on both sides of the exchange
template <int DK, bool KDA>
__device__ __forceinline__ void state_qdq(float2 (&s)[2][DK / 16], int codec, BwdSmem<DK, KDA>& sm, int warp,
                                          int lane, int rg, int cg) {
  constexpr int RPT = DK / 8, NPR = RPT / 2;
  const int r0 = RPT * rg;
  if (codec == 2) {
#pragma unroll
    for (int j = 0; j < NPR; ++j) {
      float m0 = fmaxf(fabsf(s[0][j].x), fabsf(s[1][j].x)), m1 = fmaxf(fabsf(s[0][j].y), fabsf(s[1][j].y));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      if (cg == 0) {
        sm.rmax[warp][r0 + 2 * j] = m0;
        sm.rmax[warp][r0 + 2 * j + 1] = m1;
      }
    }
    __syncthreads();
    const int w0 = warp & ~3;
    auto rowmax = [&](int row) {
      return fmaxf(fmaxf(sm.rmax[w0][row], sm.rmax[w0 + 1][row]), fmaxf(sm.rmax[w0 + 2][row], sm.rmax[w0 + 3][row]));
    };
#pragma unroll
    for (int j = 0; j < NPR; ++j) {
      const float sa = int8_scale(rowmax(r0 + 2 * j)), sb = int8_scale(rowmax(r0 + 2 * j + 1));
      const float ra = __frcp_rn(sa), rb = __frcp_rn(sb);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        s[c][j] = make_float2(int8_qdq_rcp(s[c][j].x, ra, sa), int8_qdq_rcp(s[c][j].y, rb, sb));
    }
  } else {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < NPR; ++j)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(s[0][j].x), fabsf(s[0][j].y)), fmaxf(fabsf(s[1][j].x), fabsf(s[1][j].y))));
    amax = warp_max(amax);
    if (lane == 0) sm.wmax[warp] = amax;
    __syncthreads();
    float tmax = sm.wmax[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) tmax = fmaxf(tmax, sm.wmax[w]);
    const float sc = qdq_scale(tmax), rc = __frcp_rn(sc);
    const float2 sc2 = bcast(sc), rc2 = bcast(rc);
#pragma unroll
    for (int j = 0; j < NPR; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const __nv_fp8x2_e4m3 q(__fmul2_rn(s[c][j], rc2));
        s[c][j] = __fmul2_rn(static_cast<float2>(q), sc2);
      }
  }
  __syncthreads();   // the next QDQ's shared-memory writes come after every thread's reads
}

// Slot of key row `row` in a warp's row-sum array: rows r0 .. r0 + dk / 8 - 1 of row group rg are
// permuted by xor with rg, so the stores of the 8 row groups (one row each) and the loads of 8
// consecutive rows both fall in distinct banks.
template <int DK>
__device__ __forceinline__ int rs_slot(int row) {
  constexpr int RPT = DK / 8;
  const int g = row / RPT;
  return RPT * g + ((row - RPT * g) ^ g);
}

// One token backward (header formulas) from P, the state before the token, with dS in ds (updated
// to dS_{t-1}). Writes dv; leaves the token's four row sums of every key row in sm.rs[buf] and,
// after the barrier, the reducing threads (the first dk) write the slab partials.
template <int DK, bool KDA>
__device__ __forceinline__ void bwd_token(const BwdParams& p, BwdSmem<DK, KDA>& sm, const float2 (&P)[2][DK / 16],
                                          float2 (&ds)[2][DK / 16], const TokView<DK>& t, const unsigned char* rec,
                                          int64_t tok, int h, int slab, int buf, int warp, int lane, int rg, int cg,
                                          int c0) {
  constexpr int RPT = DK / 8, NPR = RPT / 2;
  float2 pp[2][NPR];   // P' = a o P
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < NPR; ++j) {
    pp[0][j] = __fmul2_rn(P[0][j], t.a2[j]);
    pp[1][j] = __fmul2_rn(P[1][j], t.a2[j]);
    acc0 = __ffma2_rn(pp[0][j], t.k2[j], acc0);
    acc1 = __ffma2_rn(pp[1][j], t.k2[j], acc1);
  }
  // u = v - P'^T k
  float2 u = col_sum(acc0, acc1);
  u = make_float2(t.vv.x - u.x, t.vv.y - u.y);
  // dS += scale q do^T; du = b dS^T k
  const float2 sdo0 = bcast(p.scale * t.dov.x), sdo1 = bcast(p.scale * t.dov.y);
  acc0 = make_float2(0.f, 0.f);
  acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < NPR; ++j) {
    ds[0][j] = __ffma2_rn(t.q2[j], sdo0, ds[0][j]);
    ds[1][j] = __ffma2_rn(t.q2[j], sdo1, ds[1][j]);
    acc0 = __ffma2_rn(ds[0][j], t.k2[j], acc0);
    acc1 = __ffma2_rn(ds[1][j], t.k2[j], acc1);
  }
  float2 du = col_sum(acc0, acc1);
  du = make_float2(t.b * du.x, t.b * du.y);
  if (rg == 0) *reinterpret_cast<float2*>(p.grad_v + (tok * p.Hv + h) * p.dv + slab * SL + c0) = du;
  // per key-row pair, over this lane's 2 columns: X0 = S do (S = P' + b k u^T), X1 = dS u, X2 = P' du,
  // X3 = dP' . P' with dP' = dS - k du^T; then a reduce-scatter over the lane quad leaves the quad's
  // sum of X_cg in lane cg
  const float2 bu0 = bcast(t.b * u.x), bu1 = bcast(t.b * u.y);
  const float2 do0 = bcast(t.dov.x), do1 = bcast(t.dov.y);
  const float2 u0 = bcast(u.x), u1 = bcast(u.y);
  const float2 du0 = bcast(du.x), du1 = bcast(du.y), ndu0 = bcast(-du.x), ndu1 = bcast(-du.y);
  const bool hi = (cg & 2) != 0, lo = (cg & 1) != 0;
  float* rsb = reinterpret_cast<float*>(&sm.rs[buf][warp][0]);
  const int r0 = RPT * rg;
#pragma unroll
  for (int j = 0; j < NPR; ++j) {
    const float2 S0 = __ffma2_rn(t.k2[j], bu0, pp[0][j]), S1 = __ffma2_rn(t.k2[j], bu1, pp[1][j]);
    const float2 X0 = __ffma2_rn(S1, do1, __fmul2_rn(S0, do0));
    const float2 X1 = __ffma2_rn(ds[1][j], u1, __fmul2_rn(ds[0][j], u0));
    const float2 X2 = __ffma2_rn(pp[1][j], du1, __fmul2_rn(pp[0][j], du0));
    const float2 dp0 = __ffma2_rn(t.k2[j], ndu0, ds[0][j]), dp1 = __ffma2_rn(t.k2[j], ndu1, ds[1][j]);
    // dg = (dL/da) a = <dP', P> a = <dP', P'> (per key row for KDA)
    const float2 X3 = __ffma2_rn(dp1, pp[1][j], __fmul2_rn(dp0, pp[0][j]));
    ds[0][j] = __fmul2_rn(t.a2[j], dp0);   // dS_{t-1}
    ds[1][j] = __fmul2_rn(t.a2[j], dp1);
    const float2 s0 = hi ? X0 : X2, s1 = hi ? X1 : X3;
    float2 k0 = hi ? X2 : X0, k1 = hi ? X3 : X1;
    k0 = __fadd2_rn(k0, make_float2(__shfl_xor_sync(0xffffffffu, s0.x, 2), __shfl_xor_sync(0xffffffffu, s0.y, 2)));
    k1 = __fadd2_rn(k1, make_float2(__shfl_xor_sync(0xffffffffu, s1.x, 2), __shfl_xor_sync(0xffffffffu, s1.y, 2)));
    const float2 sn = lo ? k0 : k1;
    float2 r = lo ? k1 : k0;
    r = __fadd2_rn(r, make_float2(__shfl_xor_sync(0xffffffffu, sn.x, 1), __shfl_xor_sync(0xffffffffu, sn.y, 1)));
    rsb[rs_slot<DK>(r0 + 2 * j) * 4 + cg] = r.x;
    rsb[rs_slot<DK>(r0 + 2 * j + 1) * 4 + cg] = r.y;
  }
  __syncthreads();
  // per key row cr (threads cr < DK): the slab's sums over its warps, in warp order
  if (threadIdx.x < DK) {
    const int cr = threadIdx.x, slot = rs_slot<DK>(cr);
    float4 a = sm.rs[buf][0][slot];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      const float4 x = sm.rs[buf][w][slot];
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    }
    const int64_t ph = (int64_t)slab * p.tokens * p.Hv + tok * p.Hv + h;   // slab partial index of (tok, h)
    p.part_q[ph * DK + cr] = p.scale * a.x;
    p.part_k[ph * DK + cr] = t.b * a.y - a.z;
    if (KDA) p.part_g[ph * DK + cr] = a.w;
    const float kc = bf16_to_f32(reinterpret_cast<const __nv_bfloat16*>(rec + Rec<DK, KDA>::K)[cr]);
    // db = sum over key rows of k (dS u); GDN dg = sum over key rows of dP' . P'
    const float db = warp_sum(kc * a.y);
    const float dg = KDA ? 0.f : warp_sum(a.w);
    if (lane == 0) {
      const int64_t pw = ((int64_t)slab * (DK / 32) + warp) * p.tokens * p.Hv + tok * p.Hv + h;
      p.part_b[pw] = db;
      if (!KDA) p.part_g[pw] = dg;
    }
  }
}

template <int DK, bool KDA>
__global__ void __launch_bounds__(NT, 1) chunk_bwd_kernel(const BwdParams p) {
  constexpr int RPT = DK / 8, NPR = RPT / 2;
  using R = Rec<DK, KDA>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem<DK, KDA>& sm = *reinterpret_cast<BwdSmem<DK, KDA>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = lane >> 2, cg = lane & 3;
  const int c0 = warp * 8 + cg * 2;   // this lane's first column within the slab
  const int r0 = RPT * rg;            // this lane's first key row
  const int nslab = p.dv / SL;
  const int64_t units = (int64_t)p.N * p.Hv * nslab;
  float2* const scr = reinterpret_cast<float2*>(p.scratch) + (int64_t)blockIdx.x * NSUB * RPT * NT;
  // thread-major copies of a register state: element (c, j) of sub-chunk checkpoint q / slot m
  auto sub_at = [&](int q, int c, int j) { return scr + ((int64_t)q * RPT + c * NPR + j) * NT + tid; };
  auto slot_at = [&](int m, int c, int j) { return &sm.slot[m][c * NPR + j][tid]; };
  int tc = 0;   // backward tokens so far (selects the row-sum buffer)

  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int slab = (int)(unit % nslab);
    const int64_t nh = unit / nslab;   // n * Hv + h
    const int n = (int)(nh / p.Hv), h = (int)(nh % p.Hv);
    const int hq = h / (p.Hv / p.Hqk);
    const int col = slab * SL + c0;    // this lane's first value column
    const int64_t t0 = p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
    const int64_t len = p.cu ? (int64_t)p.cu[n + 1] - t0 : (int64_t)p.T;
    const int64_t nch = (len + kChunk - 1) / kChunk;
    const int64_t slot0 = t0 / kChunk + n;
    const int64_t st = (int64_t)DK * p.dv;   // one state
    auto ck = [&](int64_t c) { return p.ckpt + ((slot0 + c) * p.Hv + h) * st; };
    TokView<DK> tv;

    // ---- pass 1: the forward recurrence, storing the state entering every chunk; the tokens
    // stream through the two halves of the staging area, 32 at a time ----
    float2 s[2][NPR];
    if (p.h0) {
      load_state<DK>(s, p.h0 + nh * st, p.dv, r0, col);
    } else {
#pragma unroll
      for (int j = 0; j < NPR; ++j) s[0][j] = s[1][j] = make_float2(0.f, 0.f);
    }
    const int64_t nblk = (len + 31) / 32;
    __syncthreads();   // the previous unit's last reads of the staging area are done
    for (int64_t b = 0; b < 2 && b < nblk; ++b) {
      stage_tokens<DK, KDA>(p, sm.stage + b * 32 * R::BYTES, t0 + 32 * b, (int)min((int64_t)32, len - 32 * b), h,
                            hq, slab);
      cp_commit();
    }
    for (int64_t b = 0; b < nblk; ++b) {
      if (b + 1 < nblk) cp_wait<1>(); else cp_wait<0>();
      __syncthreads();
      unsigned char* half = sm.stage + (b & 1) * 32 * R::BYTES;
      const int nb = (int)min((int64_t)32, len - 32 * b);
      exp_gates<DK, KDA>(half, nb);
      __syncthreads();
      for (int r = 0; r < nb; ++r) {
        const int64_t t = 32 * b + r;
        if (t % kChunk == 0) store_state<DK>(s, ck(t / kChunk), p.dv, r0, col);
        read_token<DK, KDA>(half + r * R::BYTES, rg, c0, false, tv);
        fwd_step<DK>(s, tv);
        if (p.state_qdq && (t + 1) % kChunk == 0) state_qdq<DK, KDA>(s, p.state_qdq, sm, warp, lane, rg, cg);
      }
      __syncthreads();   // every thread is done with this half
      if (b + 2 < nblk) {
        stage_tokens<DK, KDA>(p, half, t0 + 32 * (b + 2), (int)min((int64_t)32, len - 32 * (b + 2)), h, hq, slab);
        cp_commit();
      }
    }

    // ---- pass 2: chunks in reverse; dS in registers ----
    float2 ds[2][NPR];
    if (p.dhT) {
      load_state<DK>(ds, p.dhT + nh * st, p.dv, r0, col);
    } else {
#pragma unroll
      for (int j = 0; j < NPR; ++j) ds[0][j] = ds[1][j] = make_float2(0.f, 0.f);
    }
    for (int64_t c = nch - 1; c >= 0; --c) {
      const int L = (int)min((int64_t)kChunk, len - c * kChunk);
      const int64_t tc0 = t0 + c * kChunk;
      __syncthreads();   // the staging area is free
      stage_tokens<DK, KDA>(p, sm.stage, tc0, L, h, hq, slab);
      cp_commit();
      cp_wait<0>();
      __syncthreads();
      exp_gates<DK, KDA>(sm.stage, L);
      __syncthreads();
      // the sub-chunk checkpoints: the state before tokens 0, 4, .., 4 (jmax - 1) to the scratch; the
      // state before token 4 jmax stays in registers
      load_state<DK>(s, ck(c), p.dv, r0, col);
      const int jmax = (L - 1) / SUB;
      for (int r = 0; r < SUB * jmax; ++r) {
        if (r % SUB == 0) {
#pragma unroll
          for (int j = 0; j < NPR; ++j) {
            *sub_at(r / SUB, 0, j) = s[0][j];
            *sub_at(r / SUB, 1, j) = s[1][j];
          }
        }
        read_token<DK, KDA>(sm.stage + r * R::BYTES, rg, c0, false, tv);
        fwd_step<DK>(s, tv);
      }
      for (int q = jmax; q >= 0; --q) {
        if (q < jmax) {
#pragma unroll
          for (int j = 0; j < NPR; ++j) {
            s[0][j] = *sub_at(q, 0, j);
            s[1][j] = *sub_at(q, 1, j);
          }
        }
        const int rq = SUB * q, cnt = min(SUB, L - rq);
        // the states before tokens rq .. rq + cnt - 2 into this thread's slots; s ends as the state
        // before the sub-chunk's last token
        for (int m = 0; m + 1 < cnt; ++m) {
#pragma unroll
          for (int j = 0; j < NPR; ++j) {
            *slot_at(m, 0, j) = s[0][j];
            *slot_at(m, 1, j) = s[1][j];
          }
          read_token<DK, KDA>(sm.stage + (rq + m) * R::BYTES, rg, c0, false, tv);
          fwd_step<DK>(s, tv);
        }
        for (int m = cnt - 1; m >= 0; --m) {
          float2 P[2][NPR];
          if (m == cnt - 1) {
#pragma unroll
            for (int j = 0; j < NPR; ++j) {
              P[0][j] = s[0][j];
              P[1][j] = s[1][j];
            }
          } else {
#pragma unroll
            for (int j = 0; j < NPR; ++j) {
              P[0][j] = *slot_at(m, 0, j);
              P[1][j] = *slot_at(m, 1, j);
            }
          }
          const unsigned char* rec = sm.stage + (rq + m) * R::BYTES;
          read_token<DK, KDA>(rec, rg, c0, true, tv);
          bwd_token<DK, KDA>(p, sm, P, ds, tv, rec, tc0 + rq + m, h, slab, tc & 1, warp, lane, rg, cg, c0);
          ++tc;
        }
      }
    }
    if (p.dh0) store_state<DK>(ds, p.dh0 + nh * st, p.dv, r0, col);
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

// The same sums, four consecutive outputs per thread as float4 (when inner is a multiple of 4, or
// inner = G = 1, the four sources of every term are consecutive; sizes, strides and the output
// are 16-byte aligned), each output summed in the same order as above.
__global__ void sum_parts4_kernel(const float4* __restrict__ part, float4* __restrict__ out, int64_t n_out4, int nslab,
                                  int64_t slab_stride4, int G, int inner4) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_out4; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t base = (e / inner4) * G * inner4 + e % inner4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nslab; ++s)
      for (int j = 0; j < G; ++j) {
        const float4 x = part[s * slab_stride4 + base + (int64_t)j * inner4];
        acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
      }
    out[e] = acc;
  }
}

constexpr int kBwdCtas = 152;   // one CTA per GB300 SM at most; each owns a sub-chunk scratch

template <int DK, bool KDA>
cudaError_t launch_t(const BwdParams& bp, int64_t units, cudaStream_t stream) {
  int dev = 0, sms = kBwdCtas;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaGetLastError();
  int64_t grid = units < (int64_t)sms ? units : (int64_t)sms;
  if (grid > kBwdCtas) grid = kBwdCtas;
  const size_t smem = sizeof(BwdSmem<DK, KDA>);
  cudaError_t e = cudaFuncSetAttribute(chunk_bwd_kernel<DK, KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  chunk_bwd_kernel<DK, KDA><<<(unsigned)grid, NT, smem, stream>>>(bp);
  return cudaGetLastError();
}

cudaError_t sum_parts(const float* part, float* out, int64_t n_out, int nslab, int64_t slab_stride, int G, int inner,
                      cudaStream_t stream) {
  if (n_out == 0) return cudaSuccess;
  const bool vec = n_out % 4 == 0 && slab_stride % 4 == 0 && (inner % 4 == 0 || (inner == 1 && G == 1)) &&
                   (reinterpret_cast<uintptr_t>(part) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  if (vec) {
    const int64_t n4 = n_out / 4, blocks = (n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16;
    sum_parts4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(part),
                                                            reinterpret_cast<float4*>(out), n4, nslab, slab_stride / 4,
                                                            G, inner == 1 ? 1 : inner / 4);
  } else {
    const int64_t blocks = (n_out + 255) / 256 < 152 * 32 ? (n_out + 255) / 256 : 152 * 32;
    sum_parts_kernel<<<(unsigned)blocks, 256, 0, stream>>>(part, out, n_out, nslab, slab_stride, G, inner);
  }
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
  const int nwr = p.dk / 32;   // reducing warps: db (and GDN dg) partials per slab
  l.off_scratch = up(l.off_ckpt + (size_t)slots * p.Hv * p.dk * p.dv * 4);
  l.off_part_q = up(l.off_scratch + (size_t)ctas * NSUB * p.dk * SL * 4);
  l.off_part_k = up(l.off_part_q + part * p.dk);
  l.off_part_b = up(l.off_part_k + part * p.dk);
  l.off_part_g = up(l.off_part_b + part * nwr);
  l.total = up(l.off_part_g + part * (p.kda ? p.dk : nwr));
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
  const int nwr = p.dk / 32;
  if ((e = sum_parts(pb, gr.dbeta, sh, nslab * nwr, sh, 1, 1, stream)) != cudaSuccess) return e;
  if (p.kda) return sum_parts(pg, gr.dg, sh * p.dk, nslab, sh * p.dk, 1, 1, stream);
  return sum_parts(pg, gr.dg, sh, nslab * nwr, sh, 1, 1, stream);
}

}  // namespace gdn
