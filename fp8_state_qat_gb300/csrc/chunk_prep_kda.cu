// chunk_prep_kda.cu -- the state-independent half of the chunked KDA forward (dk = 128): one CTA of
// 256 threads per (chunk, v-head) work item, all items in parallel.
//
// KDA keeps one retention per key channel ("Add KDA prefill numerical emulation for QAT", "What
// does this PR do?"): with gam[r][c] = prefix sums of g[.][c] inside the chunk,
//   A[r][i] = beta_r sum_c k_r[c] k_i[c] exp(gam_r[c] - gam_i[c])   (i < r)
//   P[r][i] =        sum_c q_r[c] k_i[c] exp(gam_r[c] - gam_i[c])   (i <= r)   -> workspace, hi + lo
//   T = (I + A)^{-1};  T'' = T diag(beta)                                       -> workspace, hi + lo
//   W = T'' (K o exp(gam)),  one E4M3 scale over the chunk's W (W QDQ)          -> workspace, W^T
//   Qd = Q o exp(gam),  Kd = K o exp(gam_63 - gam)                              -> workspace, hi + lo
//   exp(gam_63[c])                                                               -> workspace
// so that the state chain needs no per-channel exponentials: Y = Qd S0, C = Kd^T Delta,
// S1 = diag(exp(gam_63)) S0 + C.
//
// The pairwise decays factor through a per-channel anchor: exp(gam_r - gam_i) = exp(gam_r - m)
// exp(m - gam_i). When every channel's gam spans at most kChunkSpan over the chunk, m is the
// midpoint of its range, both factors stay within exp(+-kChunkSpan / 2) (normal in fp32 and bf16),
// and A and P are one tcgen05 product, [K o e^(gam - m) ; Q o e^(gam - m)] (K o e^(m - gam))^T, on
// bf16 hi + lo operands, masked to i < r (A) and i <= r (P). Steeper chunks take CUDA cores:
// the pairwise decays factor through the first token a = 16 b of each 16-row block b:
// exp(gam_r - gam_i) = exp(gam_r - gam_a) exp(gam_a - gam_i), so A and P for rows of block b are
// plain dot products of rows decayed to a. Below the diagonal block both exponents are <= 0 for
// log-decays g <= 0 (no overflow; a factor that underflows bounds a product that is as small).
// Inside the diagonal block exp(gam_a - gam_i) >= 1; the factored form is used there when every
// channel's |gam_i - gam_a| over the block stays <= kDiagRange (both factors normal fp32, each
// exponential's relative error a few 1e-6), else that block takes the pairwise exponentials
// directly. The WY products run on tcgen05 (bf16 hi + lo);
// the rest on CUDA cores. Every mbarrier wait is bounded; a CTA that gives up records it in the
// status word, waits (bounded) for its TMA load in flight, frees its TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t KB = 1024;
constexpr int GLD = 132;   // row stride (floats) of gam and of the decayed-row scratch
constexpr int A_LD = 68;
constexpr float kDiagRange = 40.f;
constexpr float kChunkSpan = 64.f;
// shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0, OFF_K = 16 * KB;           // Q0 | Q1, K0 | K1 (TMA, 128-byte swizzle); later W^T
constexpr uint32_t OFF_G = 32 * KB;                      // gam fp32 [64][GLD]
constexpr uint32_t OFF_A = 66 * KB;                      // A fp32 [64][A_LD]
constexpr uint32_t OFF_T = 83 * KB;                      // P fp32 [64][A_LD] (before the solve), then T
constexpr uint32_t OFF_SCR = 100 * KB;                   // 64 KB: decayed rows; solve scratch; Qd | Kd; Kt
constexpr uint32_t OFF_TT = 164 * KB;                    // T'' hi | lo [64 r][64 i] K-major
constexpr uint32_t OFF_P = 180 * KB;                     // P hi | lo [64 r][64 i] K-major
constexpr uint32_t OFF_VEC = 196 * KB;                   // beta [64], partial maxima [8], anchor m [128] at 128
// tensor-core A / P operands (bf16 hi, lo): [K o e^(gam - m) ; Q o e^(gam - m)] (128 rows, k blocks 16 KB
// apart), K o e^(m - gam) (64 rows, k blocks 8 KB apart); they overlay the scratch, T'' and P regions
constexpr uint32_t OFF_LQ = OFF_SCR, OFF_LQ_LO = OFF_SCR + 32 * KB, OFF_KR = OFF_SCR + 64 * KB, OFF_KR_LO = OFF_KR + 16 * KB;
constexpr uint32_t kSmemBytes = OFF_VEC + 1024 + 1024;   // + slack to align the base
static_assert(OFF_G + 64 * GLD * 4 <= OFF_A && OFF_A + 64 * A_LD * 4 <= OFF_T && OFF_T + 64 * A_LD * 4 <= OFF_SCR,
              "regions overlap");
static_assert((16 + 16 + 64) * GLD * 4 <= 64 * KB, "decayed-row scratch exceeds its region");
static_assert(OFF_KR_LO + 16 * KB <= OFF_VEC && OFF_TT >= OFF_KR && OFF_P >= OFF_KR_LO, "operand overlay");
static_assert(kThreads == 256, "the thread mappings below assume 256 threads");

constexpr uint32_t TM_WT = 0;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t IDESC_WT = tc::make_idesc(tc::kKindBF16, 128, 64, true, false);   // Kt^T (MN) x T''^T (K)
constexpr uint32_t IDESC_AP = tc::make_idesc(tc::kKindBF16, 128, 64, false, false);  // [Kl ; Ql] (K) x Kr (K)

struct KdaPrepParams {
  const float* g;      // [tokens, Hv, 128]
  const float* beta;   // [tokens, Hv]
  const int32_t* cu;
  float* vec;
  int* status;
  int T, N, Hqk, Hv;
  int w_qdq;
};

__device__ __forceinline__ int64_t seq_start(const KdaPrepParams& p, int n) {
  return p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
}
// 8 consecutive bf16 of row r, columns c8 .. c8 + 7 (c8 % 8 == 0) of a swizzled [64][128] tile
__device__ __forceinline__ void tile8(const unsigned char* tile, int r, int c8, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(tile + (c8 >> 6) * 8 * KB + tc::sw128(r, 2 * (c8 & 63)));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack_bf16(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
// 4 consecutive bf16 (c4 % 4 == 0)
__device__ __forceinline__ void tile4(const unsigned char* tile, int r, int c4, float* f) {
  const uint2 u = *reinterpret_cast<const uint2*>(tile + (c4 >> 6) * 8 * KB + tc::sw128(r, 2 * (c4 & 63)));
  const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_kda_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap twt, const __grid_constant__ CUtensorMap ttt,
                      const __grid_constant__ CUtensorMap tpp, const __grid_constant__ CUtensorMap tqd,
                      const __grid_constant__ CUtensorMap tkd, const KdaPrepParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;

  const int64_t item = blockIdx.x;
  const int h = (int)(item % p.Hv);
  const int64_t slot = item / p.Hv;
  int lo = 0, hi = p.N - 1;   // the sequence owning this slot: the last n with floor(cu[n] / 64) + n <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_start(p, mid) / 64 + mid <= slot) lo = mid;
    else hi = mid - 1;
  }
  const int n = lo;
  const int64_t t0 = seq_start(p, n), len = seq_start(p, n + 1) - t0;
  const int64_t c = slot - (t0 / 64 + n);
  if (c < 0 || c * 64 >= len) return;   // no chunk uses this slot (uniform across the CTA)
  const int L = (int)(len - c * 64 < 64 ? len - c * 64 : 64);
  const int hq = h / (p.Hv / p.Hqk);
  const int tok = (int)(t0 + c * 64);

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lt = tid & 31;
  const unsigned char* Qt = sm + OFF_Q;
  const unsigned char* Kt = sm + OFF_K;
  float* const gam = reinterpret_cast<float*>(sm + OFF_G);
  float* const Am = reinterpret_cast<float*>(sm + OFF_A);
  float* const Tm = reinterpret_cast<float*>(sm + OFF_T);
  float* const scr = reinterpret_cast<float*>(sm + OFF_SCR);
  float* const vbeta = reinterpret_cast<float*>(sm + OFF_VEC);
  float* const red = vbeta + 64;
  float* const gmid = vbeta + 128;
  const uint32_t bar_k = tc::smem_u32(&bars[0]), bar_w = tc::smem_u32(&bars[1]);

  if (tid == 0) {
    tc::mbar_init(bar_k, 1);
    tc::mbar_init(bar_w, 1);
    tc::mbar_fence_init();
    tc::mbar_expect_tx(bar_k, 32 * KB);
    tc::tma_load_3d(sbase + OFF_Q, &tq, bar_k, 0, hq, tok);
    tc::tma_load_3d(sbase + OFF_Q + 8 * KB, &tq, bar_k, 64, hq, tok);
    tc::tma_load_3d(sbase + OFF_K, &tk, bar_k, 0, hq, tok);
    tc::tma_load_3d(sbase + OFF_K + 8 * KB, &tk, bar_k, 64, hq, tok);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  {   // g of the chunk (rows beyond L are zero; all loads in flight before the first store), beta
    float4 gv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + j * kThreads, r = e >> 5, c4 = (e & 31) * 4;
      gv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < L) gv[j] = __ldcs(reinterpret_cast<const float4*>(p.g + ((int64_t)(tok + r) * p.Hv + h) * 128 + c4));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + j * kThreads, r = e >> 5, c4 = (e & 31) * 4;
      *reinterpret_cast<float4*>(gam + r * GLD + c4) = gv[j];
    }
  }
  if (tid < 64) vbeta[tid] = tid < L ? p.beta[(int64_t)(tok + tid) * p.Hv + h] : 0.f;
  for (int e = tid; e < 2 * 64 * A_LD; e += kThreads) (e < 64 * A_LD ? Am : Tm)[e % (64 * A_LD)] = 0.f;
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // prefix sums per key channel, in token order; exp(gam_63) for the chain; the range of each
  // channel's gam over the chunk: its midpoint is the anchor, its width picks the A / P form
  bool steep = false;
  if (tid < 128) {
    float acc = 0.f, mx = -INFINITY, mn = INFINITY;
#pragma unroll 8
    for (int r = 0; r < 64; ++r) {
      acc += gam[r * GLD + tid];
      gam[r * GLD + tid] = acc;
      mx = fmaxf(mx, acc);
      mn = fminf(mn, acc);
    }
    p.vec[item * 256 + tid] = __expf(acc);
    gmid[tid] = 0.5f * (mx + mn);
    steep = !(mx - mn <= kChunkSpan);
  }
  const bool tc_ap = !__syncthreads_or(steep);   // uniform across the CTA
  uint32_t w_phase = 0;                           // bar_w completions waited for so far

  bool ok = true, k_done = false;
  float sW = 1.f;
  do {
    if (warp == 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_k, 0));
    if (__syncthreads_or(!ok)) break;
    k_done = true;

    if (tc_ap) {
      // ---- A and P on tcgen05 ----
      for (int t = tid; t < 64 * 16; t += kThreads) {
        const int r = t >> 4, c8 = (t & 15) * 8;
        float kf[8], qf[8], kl[8], ql[8], kr[8];
        tile8(Kt, r, c8, kf);
        tile8(Qt, r, c8, qf);
        const float4 g0 = *reinterpret_cast<const float4*>(gam + r * GLD + c8);
        const float4 g1 = *reinterpret_cast<const float4*>(gam + r * GLD + c8 + 4);
        const float4 m0 = *reinterpret_cast<const float4*>(gmid + c8);
        const float4 m1 = *reinterpret_cast<const float4*>(gmid + c8 + 4);
        const float x[8] = {g0.x - m0.x, g0.y - m0.y, g0.z - m0.z, g0.w - m0.w,
                            g1.x - m1.x, g1.y - m1.y, g1.z - m1.z, g1.w - m1.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float el = __expf(x[u]), er = __expf(-x[u]);
          kl[u] = kf[u] * el;
          ql[u] = qf[u] * el;
          kr[u] = kf[u] * er;
        }
        const uint32_t kb = (uint32_t)(c8 >> 6), col = 2 * (c8 & 63);
        const uint32_t sk = tc::sw128(r, col), sq = tc::sw128(64 + r, col);
        uint4 h16, l16;
        split8(kl, h16, l16);
        st16(sm, OFF_LQ + kb * 16 * KB + sk, h16);
        st16(sm, OFF_LQ_LO + kb * 16 * KB + sk, l16);
        split8(ql, h16, l16);
        st16(sm, OFF_LQ + kb * 16 * KB + sq, h16);
        st16(sm, OFF_LQ_LO + kb * 16 * KB + sq, l16);
        split8(kr, h16, l16);
        st16(sm, OFF_KR + kb * 8 * KB + sk, h16);
        st16(sm, OFF_KR_LO + kb * 8 * KB + sk, l16);
      }
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc::tc_fence_after();
        const uint64_t dA = tc::make_sdesc(sbase + OFF_LQ, 16, 1024);
        const uint64_t dB = tc::make_sdesc(sbase + OFF_KR, 16, 1024);
        // hi x hi + hi x lo + lo x hi
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + TM_WT, dadv(dA, (q == 2 ? 32 * KB : 0) + (ks >> 2) * 16 * KB + (ks & 3) * 32),
                         dadv(dB, (q == 1 ? 16 * KB : 0) + (ks >> 2) * 8 * KB + (ks & 3) * 32), IDESC_AP, (q | ks) != 0);
        tc::mma_commit(bar_w);
      }
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_w, w_phase & 1));
      ++w_phase;
      if (__syncthreads_or(!ok)) break;
      tc::tc_fence_after();
      if (warp < 4) {   // TMEM lane = tid: rows 0-63 give A, rows 64-127 give P
        float d[64];
        ld32(tmem, (uint32_t)warp * 32u, TM_WT, d);
        ld32(tmem, (uint32_t)warp * 32u, TM_WT + 32, d + 32);
        if (tid < 64) {
          const float br = vbeta[tid];
#pragma unroll
          for (int i = 0; i < 64; i += 4)
            *reinterpret_cast<float4*>(Am + tid * A_LD + i) =
                make_float4(i < tid ? br * d[i] : 0.f, i + 1 < tid ? br * d[i + 1] : 0.f,
                            i + 2 < tid ? br * d[i + 2] : 0.f, i + 3 < tid ? br * d[i + 3] : 0.f);
        } else {
          const int r = tid - 64;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float pv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pv[u] = 8 * q + u <= r ? d[8 * q + u] : 0.f;
            uint4 h16, l16;
            split8(pv, h16, l16);
            st16(sm, OFF_P + tc::sw128(r, 16 * q), h16);
            st16(sm, OFF_P + 8 * KB + tc::sw128(r, 16 * q), l16);
          }
        }
      }
      tc::tc_fence_before();
      __syncthreads();
    } else {
      // ---- A and P, one 16-row block b at a time ----
      float* const Rk = scr;                 // [16][GLD]: k_r exp(gam_r - gam_a), rows of block b
      float* const Rq = scr + 16 * GLD;      // [16][GLD]: q_r exp(gam_r - gam_a)
      float* const Ki = scr + 32 * GLD;      // [64][GLD]: k_i exp(gam_a - gam_i), i < a (+ 16 when factored)
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        const int a = 16 * b;
        float dev = 0.f;   // largest |gam_i - gam_a| over the block's rows and channels
        for (int e = tid; e < 16 * 128; e += kThreads) {
          const int i = a + (e >> 7), c = e & 127;
          dev = fmaxf(dev, fabsf(gam[i * GLD + c] - gam[a * GLD + c]));
        }
        const bool pairwise = __syncthreads_or(!(dev <= kDiagRange));   // uniform across the CTA
        const int nblk = pairwise ? b : b + 1;                          // column blocks as dot products
        {   // decayed rows of block b (one 8-column group per thread)
          const int rr = tid >> 4, c8 = (tid & 15) * 8;
          float kf[8], qf[8];
          tile8(Kt, a + rr, c8, kf);
          tile8(Qt, a + rr, c8, qf);
          float e[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) e[u] = __expf(gam[(a + rr) * GLD + c8 + u] - gam[a * GLD + c8 + u]);
#pragma unroll
          for (int u = 0; u < 8; u += 4) {
            *reinterpret_cast<float4*>(Rk + rr * GLD + c8 + u) =
                make_float4(kf[u] * e[u], kf[u + 1] * e[u + 1], kf[u + 2] * e[u + 2], kf[u + 3] * e[u + 3]);
            *reinterpret_cast<float4*>(Rq + rr * GLD + c8 + u) =
                make_float4(qf[u] * e[u], qf[u + 1] * e[u + 1], qf[u + 2] * e[u + 2], qf[u + 3] * e[u + 3]);
          }
        }
        for (int t = tid; t < nblk * 256; t += kThreads) {   // decayed columns i < 16 nblk
          const int i = t >> 4, c8 = (t & 15) * 8;
          float kf[8];
          tile8(Kt, i, c8, kf);
#pragma unroll
          for (int u = 0; u < 8; u += 4) {
            float4 v;
            v.x = kf[u] * __expf(gam[a * GLD + c8 + u] - gam[i * GLD + c8 + u]);
            v.y = kf[u + 1] * __expf(gam[a * GLD + c8 + u + 1] - gam[i * GLD + c8 + u + 1]);
            v.z = kf[u + 2] * __expf(gam[a * GLD + c8 + u + 2] - gam[i * GLD + c8 + u + 2]);
            v.w = kf[u + 3] * __expf(gam[a * GLD + c8 + u + 3] - gam[i * GLD + c8 + u + 3]);
            *reinterpret_cast<float4*>(Ki + i * GLD + c8 + u) = v;
          }
        }
        __syncthreads();
        if (nblk > 0) {   // dot products of decayed rows: row a + rr, columns ii + 16 m, m < nblk
          const int rr = tid >> 4, ii = tid & 15;
          float accA[4] = {0.f, 0.f, 0.f, 0.f}, accP[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
          for (int c4 = 0; c4 < 128; c4 += 4) {
            const float4 rk = *reinterpret_cast<const float4*>(Rk + rr * GLD + c4);
            const float4 rq = *reinterpret_cast<const float4*>(Rq + rr * GLD + c4);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              if (m < nblk) {
                const float4 ki = *reinterpret_cast<const float4*>(Ki + (ii + 16 * m) * GLD + c4);
                accA[m] = fmaf(rk.x, ki.x, fmaf(rk.y, ki.y, fmaf(rk.z, ki.z, fmaf(rk.w, ki.w, accA[m]))));
                accP[m] = fmaf(rq.x, ki.x, fmaf(rq.y, ki.y, fmaf(rq.z, ki.z, fmaf(rq.w, ki.w, accP[m]))));
              }
            }
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (m < nblk) {
              const int r = a + rr, i = ii + 16 * m;
              if (i < r) Am[r * A_LD + i] = vbeta[r] * accA[m];   // A is strictly lower, P includes i = r
              if (i <= r) Tm[r * A_LD + i] = accP[m];
            }
          }
        }
        if (pairwise) {   // diagonal block with a steep decay: pairs i <= r, exponentials taken pairwise
#pragma unroll 1
          for (int pr = warp; pr < 136; pr += kThreads / 32) {
            int ri = 0;
            while ((ri + 1) * (ri + 2) / 2 <= pr) ++ri;   // pair pr -> (ri, ii) with ii <= ri
            const int ii = pr - ri * (ri + 1) / 2;
            const int r = a + ri, i = a + ii, c4 = lt * 4;
            float kr[4], ki[4], qr[4];
            tile4(Kt, r, c4, kr);
            tile4(Kt, i, c4, ki);
            tile4(Qt, r, c4, qr);
            float sA = 0.f, sP = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float e = __expf(gam[r * GLD + c4 + u] - gam[i * GLD + c4 + u]);
              sA = fmaf(kr[u] * ki[u], e, sA);
              sP = fmaf(qr[u] * ki[u], e, sP);
            }
            sA = warp_sum(sA);
            sP = warp_sum(sP);
            if (lt == 0) {
              Am[r * A_LD + i] = ii < ri ? vbeta[r] * sA : 0.f;
              Tm[r * A_LD + i] = sP;
            }
          }
        }
        __syncthreads();
      }
      // P -> bf16 hi | lo, K-major [r][i] (P is read from the T region, which the solve reuses)
      for (int t = tid; t < 512; t += kThreads) {
        const int r = t >> 3, i0 = (t & 7) * 8;
        const float4 pa = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0);
        const float4 pb = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0 + 4);
        const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        uint4 h16, l16;
        split8(pv, h16, l16);
        const uint32_t off = tc::sw128(r, 2 * i0);
        st16(sm, OFF_P + off, h16);
        st16(sm, OFF_P + 8 * KB + off, l16);
      }
      __syncthreads();
      for (int e = tid; e < 64 * A_LD; e += kThreads) Tm[e] = 0.f;
      __syncthreads();
    }

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then the blocks below
    // the diagonal by levels of T_ij = -T_ii sum_{j <= m < i} A_im T_mj ----
    if (tid < 64) {
      const int b0 = (tid >> 4) * 16, jj = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const float* arow = Am + (b0 + r) * A_LD + b0;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) {
          const float t = arow[i] * x[i];
          if ((i & 3) == 0) a0 += t;
          else if ((i & 3) == 1) a1 += t;
          else if ((i & 3) == 2) a2 += t;
          else a3 += t;
        }
        const float acc = ((r == jj) ? 1.f : 0.f) - ((a0 + a1) + (a2 + a3));
        x[r] = r < jj ? 0.f : acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) Tm[(b0 + r) * A_LD + b0 + jj] = x[r];
    }
    __syncthreads();
    {
      // one 1 x 4 tile (row rr, columns c4 .. c4 + 3) of a 16 x 16 block per thread
      const int blk = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
      auto ytile = [&](int bi, int bj, float* y) {
        y[0] = y[1] = y[2] = y[3] = 0.f;
#pragma unroll 4
        for (int m = 0; m < 16 * (bi - bj); ++m) {
          const float a = Am[(bi * 16 + rr) * A_LD + bj * 16 + m];
          const float4 t = *reinterpret_cast<const float4*>(Tm + (bj * 16 + m) * A_LD + bj * 16 + c4);
          y[0] = fmaf(a, t.x, y[0]); y[1] = fmaf(a, t.y, y[1]); y[2] = fmaf(a, t.z, y[2]); y[3] = fmaf(a, t.w, y[3]);
        }
      };
      auto ttile = [&](int bi, int bj, const float* Y) {
        float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int m = 0; m < 16; ++m) {
          const float a = Tm[(bi * 16 + rr) * A_LD + bi * 16 + m];
          const float4 y = *reinterpret_cast<const float4*>(Y + m * 16 + c4);
          t4[0] = fmaf(a, y.x, t4[0]); t4[1] = fmaf(a, y.y, t4[1]); t4[2] = fmaf(a, y.z, t4[2]); t4[3] = fmaf(a, y.w, t4[3]);
        }
        *reinterpret_cast<float4*>(Tm + (bi * 16 + rr) * A_LD + bj * 16 + c4) = make_float4(-t4[0], -t4[1], -t4[2], -t4[3]);
      };
      auto put = [&](float* Y, const float* y) { *reinterpret_cast<float4*>(Y + rr * 16 + c4) = make_float4(y[0], y[1], y[2], y[3]); };
      float y[4];
      if (blk < 3) { ytile(blk + 1, blk, y); put(scr + blk * 256, y); }   // level 1: (1,0) (2,1) (3,2)
      __syncthreads();
      if (blk < 3) ttile(blk + 1, blk, scr + blk * 256);
      __syncthreads();
      if (blk < 2) { ytile(blk + 2, blk, y); put(scr + blk * 256, y); }   // level 2: (2,0) (3,1)
      __syncthreads();
      if (blk < 2) ttile(blk + 2, blk, scr + blk * 256);
      __syncthreads();
      if (blk == 0) { ytile(3, 0, y); put(scr, y); }                       // level 3: (3,0)
      __syncthreads();
      if (blk == 0) ttile(3, 0, scr);
      __syncthreads();
    }

    // ---- T'' = T diag(beta) (hi | lo, K-major [r][i]); Qd, Kd (hi | lo, [row][c] in 64-column blocks) ----
    for (int t = tid; t < 512; t += kThreads) {
      const int r = t >> 3, i0 = (t & 7) * 8;
      const float4 ta = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0);
      const float4 tb = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0 + 4);
      const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
      float t2[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) t2[u] = tv[u] * vbeta[i0 + u];
      uint4 h16, l16;
      split8(t2, h16, l16);
      const uint32_t off = tc::sw128(r, 2 * i0);
      st16(sm, OFF_TT + off, h16);
      st16(sm, OFF_TT + 8 * KB + off, l16);
    }
    for (int t = tid; t < 64 * 16; t += kThreads) {
      const int r = t >> 4, c8 = (t & 15) * 8;
      float qf[8], kf[8], xq[8], xk[8];
      tile8(Qt, r, c8, qf);
      tile8(Kt, r, c8, kf);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float gr = gam[r * GLD + c8 + u];
        xq[u] = qf[u] * __expf(gr);
        xk[u] = kf[u] * __expf(gam[63 * GLD + c8 + u] - gr);
      }
      const uint32_t off = (c8 >> 6) * 8 * KB + tc::sw128(r, 2 * (c8 & 63));
      uint4 h16, l16;
      split8(xq, h16, l16);
      st16(sm, OFF_SCR + off, h16);
      st16(sm, OFF_SCR + 16 * KB + off, l16);
      split8(xk, h16, l16);
      st16(sm, OFF_SCR + 32 * KB + off, h16);
      st16(sm, OFF_SCR + 48 * KB + off, l16);
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tma_store_2d(&ttt, sbase + OFF_TT, 0, (int)(item * 128));
      tc::tma_store_2d(&tpp, sbase + OFF_P, 0, (int)(item * 128));
      tc::tma_store_2d(&tqd, sbase + OFF_SCR, 0, (int)(item * 256));
      tc::tma_store_2d(&tqd, sbase + OFF_SCR + 16 * KB, 0, (int)(item * 256 + 128));
      tc::tma_store_2d(&tkd, sbase + OFF_SCR + 32 * KB, 0, (int)(item * 256));
      tc::tma_store_2d(&tkd, sbase + OFF_SCR + 48 * KB, 0, (int)(item * 256 + 128));
      tc::bulk_commit();
      tc::bulk_wait_read();   // the scratch is rewritten below
    }
    __syncthreads();
    // K o exp(gam) (hi | lo): the MN-major operand of W^T = (K o exp(gam))^T T''^T
    for (int t = tid; t < 64 * 16; t += kThreads) {
      const int r = t >> 4, c8 = (t & 15) * 8;
      float kf[8], xk[8];
      tile8(Kt, r, c8, kf);
#pragma unroll
      for (int u = 0; u < 8; ++u) xk[u] = kf[u] * __expf(gam[r * GLD + c8 + u]);
      const uint32_t off = (c8 >> 6) * 8 * KB + tc::sw128(r, 2 * (c8 & 63));
      uint4 h16, l16;
      split8(xk, h16, l16);
      st16(sm, OFF_SCR + off, h16);
      st16(sm, OFF_SCR + 16 * KB + off, l16);
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      const uint64_t dA = tc::make_sdesc(sbase + OFF_SCR, 8 * KB, 1024);   // MN-major, key blocks 8 KB apart
      const uint64_t dB = tc::make_sdesc(sbase + OFF_TT, 16, 1024);        // K-major T'' [r][i]
      // Kt_hi T''_hi + Kt_hi T''_lo + Kt_lo T''_hi
#pragma unroll
      for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_WT, dadv(dA, (q == 2 ? 16 * KB : 0) + ks * 2048), dadv(dB, (q == 1 ? 8 * KB : 0) + ks * 32),
                       IDESC_WT, (q | ks) != 0);
      tc::mma_commit(bar_w);
    }
    ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_w, w_phase & 1));
    ++w_phase;
    if (__syncthreads_or(!ok)) break;
    tc::tc_fence_after();

    // ---- W QDQ: warps 0-3, thread = key channel c (TMEM lane), its 64 values W[r][c]; row c of W^T
    // goes to the Q0 slot (c < 64) or the Q1 slot ----
    float w[64];
    if (warp < 4) {
      ld32(tmem, (uint32_t)warp * 32u, TM_WT, w);
      ld32(tmem, (uint32_t)warp * 32u, TM_WT + 32, w + 32);
    }
    const uint32_t wrow = OFF_Q + (tid < 64 ? 0u : 8 * KB);
    if (p.w_qdq) {
      if (warp < 4) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) m = fmaxf(m, fabsf(w[j]));
        m = warp_max(m);
        if (lt == 0) red[warp] = m;
      }
      __syncthreads();
      const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
      sW = qdq_scale(amax);
      const float rW = __frcp_rn(sW);
      if (warp < 4) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float cd[8], dq[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2) qdq_pair(w[8 * q + u], w[8 * q + u + 1], rW, sW, cd[u], cd[u + 1], dq[u], dq[u + 1]);
          st16(sm, wrow + tc::sw128(tid & 63, 16 * q), pack8(cd));
        }
      }
    } else if (warp < 4) {   // hi -> the Q slots, lo -> the K slots
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint4 h16, l16;
        split8(w + 8 * q, h16, l16);
        st16(sm, wrow + tc::sw128(tid & 63, 16 * q), h16);
        st16(sm, wrow + 16 * KB + tc::sw128(tid & 63, 16 * q), l16);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (p.w_qdq) {
        tc::tma_store_2d(&twt, sbase + OFF_Q, 0, (int)(item * 128));
        tc::tma_store_2d(&twt, sbase + OFF_Q + 8 * KB, 0, (int)(item * 128 + 64));
      } else {
        tc::tma_store_2d(&twt, sbase + OFF_Q, 0, (int)(item * 256));
        tc::tma_store_2d(&twt, sbase + OFF_Q + 8 * KB, 0, (int)(item * 256 + 64));
        tc::tma_store_2d(&twt, sbase + OFF_K, 0, (int)(item * 256 + 128));
        tc::tma_store_2d(&twt, sbase + OFF_K + 8 * KB, 0, (int)(item * 256 + 192));
      }
      tc::bulk_commit();
      p.vec[item * 256 + 192] = sW;
    }
  } while (0);

  if (!ok && tid == 0) {
    atomicExch(p.status, 1);
    if (!k_done) tc::mbar_wait(bar_k, 0, 1u << 16);   // the Q/K tiles may still be landing
  }
  if (tid == 0) tc::bulk_wait_read();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_kda_prep(const ChunkProblem& p, const KdaLayout& lay, unsigned char* ws, cudaStream_t stream) {
  if (lay.items == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  const int64_t tmap = tokens > 0 ? tokens : 1;
  CUtensorMap tq, tk, twt, ttt, tpp, tqd, tkd;
  if (!make_bf16_map(&tq, p.q, 128, p.Hqk, tmap) || !make_bf16_map(&tk, p.k, 128, p.Hqk, tmap) ||
      !make_bf16_rows_map(&twt, ws + lay.off_wt, lay.items * (p.w_qdq ? 128 : 256), 64) ||
      !make_bf16_rows_map(&ttt, ws + lay.off_tt, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tpp, ws + lay.off_p, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tqd, ws + lay.off_qd, lay.items * 256, 128) ||
      !make_bf16_rows_map(&tkd, ws + lay.off_kd, lay.items * 256, 128))
    return cudaErrorInvalidValue;
  KdaPrepParams pp{p.g, p.beta, p.cu, reinterpret_cast<float*>(ws + lay.off_vec), reinterpret_cast<int*>(ws),
                   p.T, p.N, p.Hqk, p.Hv, p.w_qdq};
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_prep_kda_kernel<<<(unsigned)lay.items, kThreads, kSmemBytes, stream>>>(tq, tk, twt, ttt, tpp, tqd, tkd, pp);
  return cudaGetLastError();
}

}  // namespace gdn
