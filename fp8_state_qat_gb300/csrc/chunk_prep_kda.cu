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
// S1 = diag(exp(gam_63)) S0 + C. Every output goes from registers straight to global memory, in
// the row-major bf16 layout the chain kernel's TMA loads read.
//
// The pairwise decays factor through a per-channel anchor: exp(gam_r - gam_i) = exp(gam_r - m)
// exp(m - gam_i). When every channel's gam spans at most kChunkSpan over the chunk, m is the
// midpoint of its range, both factors stay within exp(+-kChunkSpan / 2) (normal in fp32 and bf16),
// and A and P are one tcgen05 product, [K o e^(gam - m) ; Q o e^(gam - m)] (K o e^(m - gam))^T, on
// bf16 hi + lo operands, masked to i < r (A) and i <= r (P); Qd, Kd and K o exp(gam) then follow
// from the same two exponentials and the per-channel factors e^m, e^(gam_63 - m). Steeper chunks
// take CUDA cores: the pairwise decays factor through the first token a = 16 b of each 16-row
// block b: exp(gam_r - gam_i) = exp(gam_r - gam_a) exp(gam_a - gam_i), so A and P for rows of
// block b are plain dot products of rows decayed to a. Below the diagonal block both exponents are
// <= 0 for log-decays g <= 0 (no overflow; a factor that underflows bounds a product that is as
// small). Inside the diagonal block exp(gam_a - gam_i) >= 1; the factored form is used there when
// every channel's |gam_i - gam_a| over the block stays <= kDiagRange (both factors normal fp32,
// each exponential's relative error a few 1e-6), else that block takes the pairwise exponentials
// directly. The WY products run on tcgen05 (bf16 hi + lo); the rest on CUDA cores. Every mbarrier
// wait is bounded; a CTA that gives up records it in the status word, waits (bounded) for its TMA
// load in flight, frees its TMEM and exits.
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
constexpr uint32_t OFF_Q = 0, OFF_K = 16 * KB;   // Q0 | Q1, K0 | K1 (TMA, 128-byte swizzle); then K o exp(gam) hi | lo
constexpr uint32_t OFF_G = 32 * KB;              // gam fp32 [64][GLD]
constexpr uint32_t OFF_A = 66 * KB;              // A fp32 [64][A_LD]
constexpr uint32_t OFF_T = 83 * KB;              // P fp32 [64][A_LD] (CUDA-core form, before the solve), then T
constexpr uint32_t OFF_SCR = 100 * KB;           // 64 KB: decayed rows (CUDA-core form); solve scratch
constexpr uint32_t OFF_TT = 164 * KB;            // T'' hi | lo [64 r][64 i] K-major
constexpr uint32_t OFF_VEC = 196 * KB;           // beta [64], partial maxima [8], then [128] each: m, e^m, e^(gam_63 - m); beta of the next item at 512
// tensor-core A / P operands (bf16 hi, lo): [K o e^(gam - m) ; Q o e^(gam - m)] (128 rows, k blocks 16 KB
// apart), K o e^(m - gam) (64 rows, k blocks 8 KB apart); they overlay the scratch and T'' regions
constexpr uint32_t OFF_LQ = OFF_SCR, OFF_LQ_LO = OFF_SCR + 32 * KB, OFF_KR = OFF_SCR + 64 * KB, OFF_KR_LO = OFF_KR + 16 * KB;
constexpr uint32_t kSmemBytes = OFF_VEC + 3 * KB + 1024;   // + slack to align the base
static_assert(OFF_G + 64 * GLD * 4 <= OFF_A && OFF_A + 64 * A_LD * 4 <= OFF_T && OFF_T + 64 * A_LD * 4 <= OFF_SCR,
              "regions overlap");
static_assert((16 + 16 + 64) * GLD * 4 <= 64 * KB, "decayed-row scratch exceeds its region");
static_assert(OFF_KR_LO + 16 * KB <= OFF_VEC && OFF_TT + 16 * KB <= OFF_VEC, "operand overlay");
static_assert(kThreads == 256, "the thread mappings below assume 256 threads");

constexpr uint32_t TM_WT = 0;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t IDESC_WT = tc::make_idesc(tc::kKindBF16, 128, 64, true, false);   // Kt^T (MN) x T''^T (K)
constexpr uint32_t IDESC_AP = tc::make_idesc(tc::kKindBF16, 128, 64, false, false);  // [Kl ; Ql] (K) x Kr (K)

struct KdaPrepParams {
  const float* g;      // [tokens, Hv, 128]
  const float* beta;   // [tokens, Hv]
  const int32_t* cu;
  const int32_t* lens; // tokens run per sequence, or null (whole sequences)
  float* vec;          // per item: exp(gam_63) [128], W scale at 192
  unsigned char* wt;   // per item 128 (W QDQ) or 256 rows of 128 bytes: W^T codes, or hi then lo
  unsigned char* tt;   // per item 128 rows: T'' hi [64 r], lo [64 r]
  unsigned char* pp;   // per item 128 rows: P hi, lo
  unsigned char* qd;   // per item 256 rows: Qd hi [c < 64: 64 r | c >= 64: 64 r], lo (same)
  unsigned char* kd;   // per item 256 rows: Kd, same layout
  int* status;
  int64_t items;
  int T, N, Hqk, Hv;
  int w_qdq;
};

// cp.async of `bytes` (4 or 16) with zero fill: src_bytes = 0 reads nothing and writes zeros
__device__ __forceinline__ void cp_async_zfill16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_zfill4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// 8 consecutive floats from shared memory (16-byte aligned)
__device__ __forceinline__ void ld8(const float* src, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// 16 bytes into column group col8 (0..7) of a 128-byte row of a workspace array
__device__ __forceinline__ void stg16(unsigned char* base, int64_t row, int col8, uint4 v) {
  *reinterpret_cast<uint4*>(base + row * 128 + col8 * 16) = v;
}

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
                      const KdaPrepParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;

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
  float* const vec_s = reinterpret_cast<float*>(sm + OFF_VEC);
  float* const red = vec_s + 64;
  float* const gmid = vec_s + 128;
  float* const gem = vec_s + 256;
  float* const ge63m = vec_s + 384;
  const uint32_t bar_k = tc::smem_u32(&bars[0]), bar_w = tc::smem_u32(&bars[1]);

  // Persistent: this CTA takes items blockIdx.x, + gridDim.x, ... that own a chunk. While one
  // item is processed, the next one's g and beta (cp.async, zero past the sequence end) and, once
  // the W product has read the K o exp(gam) tiles, its Q / K tiles (TMA) are already loading.
  struct Item { int64_t item; int h, hq, L, tok; };
  auto decode = [&](int64_t it, Item& f) -> bool {
    f.item = it;
    f.h = (int)(it % p.Hv);
    const int64_t slot = it / p.Hv;
    int lo = 0, hi = p.N - 1;   // the sequence owning this slot: the last n with floor(cu[n] / 64) + n <= slot
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seq_start(p, mid) / 64 + mid <= slot) lo = mid;
      else hi = mid - 1;
    }
    const int64_t t0 = seq_start(p, lo), len = p.lens ? (int64_t)p.lens[lo] : seq_start(p, lo + 1) - t0;
    const int64_t c = slot - (t0 / 64 + lo);
    if (c < 0 || c * 64 >= len) return false;   // no chunk uses this slot
    f.L = (int)(len - c * 64 < 64 ? len - c * 64 : 64);
    f.hq = f.h / (p.Hv / p.Hqk);
    f.tok = (int)(t0 + c * 64);
    return true;
  };
  auto next_item = [&](int64_t from, Item& f) -> bool {
    for (int64_t it = from; it < p.items; it += gridDim.x)
      if (decode(it, f)) return true;
    return false;
  };
  auto issue_qk = [&](const Item& f) {   // thread 0
    tc::mbar_expect_tx(bar_k, 32 * KB);
    tc::tma_load_3d(sbase + OFF_Q, &tq, bar_k, 0, f.hq, f.tok);
    tc::tma_load_3d(sbase + OFF_Q + 8 * KB, &tq, bar_k, 64, f.hq, f.tok);
    tc::tma_load_3d(sbase + OFF_K, &tk, bar_k, 0, f.hq, f.tok);
    tc::tma_load_3d(sbase + OFF_K + 8 * KB, &tk, bar_k, 64, f.hq, f.tok);
  };
  auto issue_g = [&](const Item& f, float* beta_dst) {   // all threads: g rows (zero past L) and beta
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + j * kThreads, r = e >> 5, c4 = (e & 31) * 4;
      const bool in = r < f.L;
      const float* src = in ? p.g + ((int64_t)(f.tok + r) * p.Hv + f.h) * 128 + c4 : p.g;
      cp_async_zfill16(gam + r * GLD + c4, src, in ? 16u : 0u);
    }
    if (tid < 64) {
      const bool in = tid < f.L;
      cp_async_zfill4(beta_dst + tid, in ? p.beta + (int64_t)(f.tok + tid) * p.Hv + f.h : p.beta, in ? 4u : 0u);
    }
  };

  if (tid == 0) {
    tc::mbar_init(bar_k, 1);
    tc::mbar_init(bar_w, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  Item cur;
  bool have = next_item(blockIdx.x, cur);
  if (have) {
    if (tid == 0) issue_qk(cur);
    issue_g(cur, vec_s + 512);
  }
  bool ok = true, k_pending = have;
  uint32_t k_phase = 0, w_phase = 0;   // completions of bar_k / bar_w waited for so far
  int vb = 1;                          // beta of the current item: vec_s + 512 vb
  while (have && ok) {
  const int64_t item = cur.item;
  float* const vbeta = vb ? vec_s + 512 : vec_s;
  Item nxt;
  const bool more = next_item(item + gridDim.x, nxt);
  cp_async_commit_wait_all();   // this item's g and beta (issued during the previous item)
  for (int e = tid; e < 2 * 64 * A_LD; e += kThreads) (e < 64 * A_LD ? Am : Tm)[e % (64 * A_LD)] = 0.f;
  __syncthreads();
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
    const float m = 0.5f * (mx + mn);
    p.vec[item * 256 + tid] = __expf(acc);
    gmid[tid] = m;
    gem[tid] = __expf(m);
    ge63m[tid] = __expf(acc - m);
    steep = !(mx - mn <= kChunkSpan);
  }
  const bool tc_ap = !__syncthreads_or(steep);   // uniform across the CTA

  // Qd, Kd (hi | lo) -> global; K o exp(gam) (hi | lo) -> smem over the Q / K tiles (each thread
  // overwrites only the tile bytes it has read); with the anchor, also the A / P operands
  auto produce = [&](bool anchored) {
    for (int t = tid; t < 64 * 16; t += kThreads) {
      const int r = t >> 4, c8 = (t & 15) * 8;
      float kf[8], qf[8], gv[8], qd[8], kd[8], kt[8];
      tile8(Qt, r, c8, qf);
      tile8(Kt, r, c8, kf);
      ld8(gam + r * GLD + c8, gv);
      const uint32_t kb = (uint32_t)(c8 >> 6), col = 2 * (c8 & 63);
      const uint32_t sk = tc::sw128(r, col);
      uint4 h16, l16;
      if (anchored) {
        float mv[8], em[8], e63[8], kl[8], ql[8], kr[8];
        ld8(gmid + c8, mv);
        ld8(gem + c8, em);
        ld8(ge63m + c8, e63);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float x = gv[u] - mv[u];
          const float el = __expf(x), er = __expf(-x);
          kl[u] = kf[u] * el;
          ql[u] = qf[u] * el;
          kr[u] = kf[u] * er;
          qd[u] = ql[u] * em[u];
          kt[u] = kl[u] * em[u];
          kd[u] = kr[u] * e63[u];
        }
        const uint32_t sq = tc::sw128(64 + r, col);
        split8(kl, h16, l16);
        st16(sm, OFF_LQ + kb * 16 * KB + sk, h16);
        st16(sm, OFF_LQ_LO + kb * 16 * KB + sk, l16);
        split8(ql, h16, l16);
        st16(sm, OFF_LQ + kb * 16 * KB + sq, h16);
        st16(sm, OFF_LQ_LO + kb * 16 * KB + sq, l16);
        split8(kr, h16, l16);
        st16(sm, OFF_KR + kb * 8 * KB + sk, h16);
        st16(sm, OFF_KR_LO + kb * 8 * KB + sk, l16);
      } else {
        float g63[8];
        ld8(gam + 63 * GLD + c8, g63);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float e1 = __expf(gv[u]), e2 = __expf(g63[u] - gv[u]);
          qd[u] = qf[u] * e1;
          kt[u] = kf[u] * e1;
          kd[u] = kf[u] * e2;
        }
      }
      const int64_t row = item * 256 + kb * 64 + r;
      const int c16 = (c8 & 63) >> 3;
      split8(qd, h16, l16);
      stg16(p.qd, row, c16, h16);
      stg16(p.qd, row + 128, c16, l16);
      split8(kd, h16, l16);
      stg16(p.kd, row, c16, h16);
      stg16(p.kd, row + 128, c16, l16);
      split8(kt, h16, l16);
      st16(sm, OFF_Q + kb * 8 * KB + sk, h16);
      st16(sm, OFF_K + kb * 8 * KB + sk, l16);
    }
  };

  float sW = 1.f;
  do {
    if (warp == 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_k, k_phase & 1));
    if (__syncthreads_or(!ok)) { ok = false; break; }
    k_pending = false;
    ++k_phase;

    if (tc_ap) {
      // ---- A and P on tcgen05 ----
      produce(true);
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (more) issue_g(nxt, vb ? vec_s : vec_s + 512);   // gam and the other beta buffer are free now
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
      if (__syncthreads_or(!ok)) { ok = false; break; }
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
            stg16(p.pp, item * 128 + r, q, h16);
            stg16(p.pp, item * 128 + 64 + r, q, l16);
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
      // P -> global, hi | lo (P is read from the T region, which the solve reuses)
      for (int t = tid; t < 512; t += kThreads) {
        const int r = t >> 3, i0 = (t & 7) * 8;
        float pv[8];
        ld8(Tm + r * A_LD + i0, pv);
        uint4 h16, l16;
        split8(pv, h16, l16);
        stg16(p.pp, item * 128 + r, i0 >> 3, h16);
        stg16(p.pp, item * 128 + 64 + r, i0 >> 3, l16);
      }
      __syncthreads();
      for (int e = tid; e < 64 * A_LD; e += kThreads) Tm[e] = 0.f;
      produce(false);   // the Q / K tiles have been read by A and P
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (more) issue_g(nxt, vb ? vec_s : vec_s + 512);
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

    // ---- T'' = T diag(beta): hi | lo, K-major [r][i], to smem (the W product) and global ----
    for (int t = tid; t < 512; t += kThreads) {
      const int r = t >> 3, i0 = (t & 7) * 8;
      float tv[8], bv[8], t2[8];
      ld8(Tm + r * A_LD + i0, tv);
      ld8(vbeta + i0, bv);
#pragma unroll
      for (int u = 0; u < 8; ++u) t2[u] = tv[u] * bv[u];
      uint4 h16, l16;
      split8(t2, h16, l16);
      const uint32_t off = tc::sw128(r, 2 * i0);
      st16(sm, OFF_TT + off, h16);
      st16(sm, OFF_TT + 8 * KB + off, l16);
      stg16(p.tt, item * 128 + r, i0 >> 3, h16);
      stg16(p.tt, item * 128 + 64 + r, i0 >> 3, l16);
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      const uint64_t dA = tc::make_sdesc(sbase + OFF_Q, 8 * KB, 1024);    // MN-major K o exp(gam), key blocks 8 KB apart
      const uint64_t dB = tc::make_sdesc(sbase + OFF_TT, 16, 1024);       // K-major T'' [r][i]
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
    if (__syncthreads_or(!ok)) { ok = false; break; }
    tc::tc_fence_after();
    if (more) {   // the K o exp(gam) tiles are read: the next item's Q / K can land there
      if (tid == 0) issue_qk(nxt);
      k_pending = true;
    }

    // ---- W QDQ: warps 0-3, thread = key channel c (TMEM lane), its 64 values W[r][c] = row c of W^T ----
    float w[64];
    if (warp < 4) {
      ld32(tmem, (uint32_t)warp * 32u, TM_WT, w);
      ld32(tmem, (uint32_t)warp * 32u, TM_WT + 32, w + 32);
    }
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
          stg16(p.wt, item * 128 + tid, q, pack8(cd));
        }
      }
    } else if (warp < 4) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint4 h16, l16;
        split8(w + 8 * q, h16, l16);
        stg16(p.wt, item * 256 + tid, q, h16);
        stg16(p.wt, item * 256 + 128 + tid, q, l16);
      }
    }
    if (tid == 0) p.vec[item * 256 + 192] = sW;
  } while (0);
  if (!ok) break;
  tc::tc_fence_before();
  __syncthreads();   // the next item rewrites smem this one still reads
  tc::tc_fence_after();
  cur = nxt;
  have = more;
  vb ^= 1;
  }

  if (!ok && tid == 0) {
    atomicExch(p.status, 1);
    if (k_pending) tc::mbar_wait(bar_k, k_phase & 1, 1u << 16);   // Q / K tiles may still be landing
  }
  cp_async_commit_wait_all();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_kda_prep(const ChunkProblem& p, const KdaLayout& lay, unsigned char* ws, cudaStream_t stream) {
  if (lay.items == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  const int64_t tmap = tokens > 0 ? tokens : 1;
  CUtensorMap tq, tk;
  if (!make_bf16_map(&tq, p.q, 128, p.Hqk, tmap) || !make_bf16_map(&tk, p.k, 128, p.Hqk, tmap))
    return cudaErrorInvalidValue;
  KdaPrepParams pp{p.g, p.beta, p.cu, p.lens, reinterpret_cast<float*>(ws + lay.off_vec), ws + lay.off_wt, ws + lay.off_tt,
                   ws + lay.off_p, ws + lay.off_qd, ws + lay.off_kd, reinterpret_cast<int*>(ws), lay.items,
                   p.T, p.N, p.Hqk, p.Hv, p.w_qdq};
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  int sms = 0, dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t grid = lay.items < sms ? lay.items : sms;   // one resident CTA per SM, each walking items
  chunk_prep_kda_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(tq, tk, pp);
  return cudaGetLastError();
}

}  // namespace gdn
