// chunk_tc.cu -- fused chunked gated-delta-rule forward on the sm_103a tensor cores (dk = 128).
//
// One CTA (256 threads) per (sequence n, value head h, 64-column value slab); the slab is one
// state-QDQ tile (all 128 key rows x 64 value columns), so its amax is CTA-local ("GDN state/W
// QAT foundation", "What does this PR do?"). The CTA walks the sequence's 64-token chunks; the
// state S0 (fp32) lives in TMEM and, as the MMA operand, in shared memory as bf16 hi + lo
// (or as exact E4M3 codes once it has been QDQ'd: codes are exact in bf16, the scale is
// applied in the epilogue).
//
// Per chunk of L <= 64 tokens (rows r >= L carry beta = g = 0, so they drop out), gam = prefix
// sums of g, Gam = exp(gam):
//   TMA      Q, K [64 x 128] and V [64 x 64] bf16 tiles (128-byte swizzle), next chunk prefetched
//   G1       [Q; K] K^T                         tcgen05 bf16, M=128 N=64 K=128 (exact products)
//   A, P     A[r][i] = beta_r exp(gam_r - gam_i) (k_r.k_i), i < r;  P[r][i] = exp(gam_r - gam_i)(q_r.k_i), i <= r
//   T        (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then the off-diagonal
//            blocks in three levels of the block recurrence (CUDA cores)
//   U        T'' V,  T'' = T diag(beta)         bf16 (T'' as hi + lo), M=64 N=64 K=64
//   W        T' K,   T' = T diag(beta Gam)      bf16 (T' as hi + lo), M=64 N=128 K=64
//   W QDQ    one E4M3 scale over the chunk's W; the codes (exact in bf16) become the operand
//   X, Y     W S0 and Q S0                      bf16, M=64 N=64 K=128
//   Delta    U - X;   Dt = exp(gam_L - gam) Delta
//   P Delta  bf16 (P and Delta as hi + lo),     M=64 N=64 K=64
//   C        K^T Dt                             bf16 (Dt as hi + lo), M=128 N=64 K=64
//   o        scale (Gam Y + P Delta)            rows r < L to global
//   S1       Gam_L S0 + C; QDQ(S1) when L == 64 (state QDQ); S1 -> TMEM and the operand
// Decays are exponentials of non-positive prefix differences with the causal mask applied
// before the exp ("Add KDA prefill numerical emulation for QAT", "What does this PR do?").
// The fused QDQ epilogues multiply by a correctly rounded reciprocal of the tile scale; this
// can differ from an exact divide by one ulp before the E4M3 rounding (the standalone
// fp8_tile_qdq divides exactly).
//
// Every mbarrier wait is bounded; a CTA whose wait gives up records it in the status word,
// waits (bounded) for its own TMA in flight, frees its TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t KB = 1024;
// shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t kStageBytes = 40 * KB;                                 // two stages
constexpr uint32_t ST_V = 0, ST_Q0 = 8 * KB, ST_K0 = 16 * KB, ST_Q1 = 24 * KB, ST_K1 = 32 * KB;
constexpr uint32_t OFF_SHI = 80 * KB, OFF_SLO = 96 * KB;   // S0 bf16 [128 c][64 j], MN-major
constexpr uint32_t OFF_TT = 112 * KB;   // T'' hi, lo, T' hi, lo (8 KB each, [r][i] K-major);
                                        // later Delta hi, lo and Dt hi, lo ([i][j] MN-major)
constexpr uint32_t OFF_P = 144 * KB;    // P hi, lo bf16 [64 r][64 i] K-major (8 KB each)
constexpr uint32_t OFF_CW = 160 * KB;   // W codes (or W hi) bf16 [64 r][128 c] K-major; W lo at +16 KB
constexpr uint32_t OFF_A = 192 * KB;    // fp32 A [64][68] (T is built in the OFF_TT region)
constexpr uint32_t A_LD = 68;
constexpr uint32_t OFF_SCR = OFF_A + 64 * A_LD * 4;   // solve scratch 3 x 16 x 16 fp32
constexpr uint32_t OFF_VEC = OFF_SCR + 16 * 48 * 4;   // 2 x {gam, Gam, decay-to-end, beta} [64] (by chunk parity)
constexpr uint32_t OFF_RED = OFF_VEC + 2 * 4 * 64 * 4;  // 8 partial maxima
constexpr uint32_t kSmemBytes = OFF_RED + 64 + 1024;  // + slack to align the base to 1024

// TMEM columns (fp32 accumulators; M=64 results use lanes 32 q + (0..15))
constexpr uint32_t TM_G1 = 0, TM_W = 64, TM_U = 192, TM_X = 256, TM_Y = 320, TM_C = 384, TM_S = 448;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t IDESC_G1 = tc::make_idesc(tc::kKindBF16, 128, 64, false, false);
constexpr uint32_t IDESC_U = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);
constexpr uint32_t IDESC_W = tc::make_idesc(tc::kKindBF16, 64, 128, false, true);
constexpr uint32_t IDESC_XY = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);
constexpr uint32_t IDESC_C = tc::make_idesc(tc::kKindBF16, 128, 64, true, true);

struct TcParams {
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;
  float* o;
  float* hT;
  int* status;
  int T, Hqk, Hv, dv;
  float scale;
  int state_qdq, w_qdq;
  float* sscale = nullptr;   // final-state QDQ scales or null (layout: ChunkProblem::state_scales)
};

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[9];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lt = tid & 31;
  const int quad = warp & 3;          // TMEM lane quadrant this warp may access
  const int half = warp >> 2;         // which half of an accumulator's columns this warp handles
  const int col0 = half * 32;         // 64-column accumulators: columns [col0, col0 + 32)
  const int lane128 = quad * 32 + lt; // row of an M=128 accumulator
  const int row64 = quad * 16 + lt;   // row of an M=64 accumulator (valid for lt < 16)

  const int nslab = p.dv / 64;
  const int slab = blockIdx.x % nslab;
  const int h = (blockIdx.x / nslab) % p.Hv;
  const int n = blockIdx.x / (nslab * p.Hv);
  const int hq = h / (p.Hv / p.Hqk);
  int64_t t0, len;
  if (p.cu) {
    t0 = p.cu[n];
    len = (int64_t)p.cu[n + 1] - t0;
  } else {
    t0 = (int64_t)n * p.T;
    len = p.T;
  }
  float* const vecs = reinterpret_cast<float*>(sm + OFF_VEC);
  float* red = reinterpret_cast<float*>(sm + OFF_RED);
  float* Am = reinterpret_cast<float*>(sm + OFF_A);
  float* scr = reinterpret_cast<float*>(sm + OFF_SCR);
  const uint32_t bar_tma0 = tc::smem_u32(&bars[0]), bar_g1 = tc::smem_u32(&bars[2]),
                 bar_u = tc::smem_u32(&bars[3]), bar_w = tc::smem_u32(&bars[4]), bar_x = tc::smem_u32(&bars[5]),
                 bar_y = tc::smem_u32(&bars[6]), bar_pd = tc::smem_u32(&bars[7]), bar_c = tc::smem_u32(&bars[8]);

  if (tid == 0) {
    for (int i = 0; i < 9; ++i) tc::mbar_init(tc::smem_u32(&bars[i]), 1);
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tq);
    tc::tma_prefetch_desc(&tk);
    tc::tma_prefetch_desc(&tv);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane0 = (uint32_t)quad * 32u;

  // operand descriptors (128-byte swizzle, 8-row groups 1024 bytes apart)
  const uint64_t dS = tc::make_sdesc(sbase + OFF_SHI, 16 * KB, 1024);     // MN-major [c][j]; lo at +16 KB
  const uint64_t dTT = tc::make_sdesc(sbase + OFF_TT, 16, 1024);          // K-major T''/T' hi, lo
  const uint64_t dDl = tc::make_sdesc(sbase + OFF_TT, 8 * KB, 1024);      // MN-major Delta / Dt hi, lo
  const uint64_t dP = tc::make_sdesc(sbase + OFF_P, 16, 1024);            // K-major P hi, lo
  const uint64_t dCW = tc::make_sdesc(sbase + OFF_CW, 16, 1024);          // K-major W codes / hi, lo
  const uint64_t dStgK[2] = {tc::make_sdesc(sbase + 0 * kStageBytes, 16, 1024),
                             tc::make_sdesc(sbase + 1 * kStageBytes, 16, 1024)};
  const uint64_t dStgM[2] = {tc::make_sdesc(sbase + 0 * kStageBytes, 16 * KB, 1024),   // MN-major K^T / V / K
                             tc::make_sdesc(sbase + 1 * kStageBytes, 16 * KB, 1024)};

  // ---- initial state: h0 (or zeros) -> TMEM S and the bf16 hi/lo operand ----
  const int64_t sb = ((int64_t)n * p.Hv + h) * 128 * p.dv + slab * 64;   // S[c][j] at sb + c dv + j
  {
    float s[32];
    if (p.h0) {
      const float4* src = reinterpret_cast<const float4*>(p.h0 + sb + (int64_t)lane128 * p.dv + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f = src[j];
        s[4 * j] = f.x; s[4 * j + 1] = f.y; s[4 * j + 2] = f.z; s[4 * j + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) s[j] = 0.f;
    }
    st32(tmem, lane0, TM_S + col0, s);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 hi, lo;
      split8(s + 8 * q, hi, lo);
      const uint32_t off = tc::sw128(lane128, 2 * (col0 + 8 * q));
      st16(sm, OFF_SHI + off, hi);
      st16(sm, OFF_SLO + off, lo);
    }
    tc::tmem_st_wait();
  }
  bool s_exact = false;   // S operand holds exact codes (one bf16 pass) with scale s_scale
  float s_scale = 1.f;
  float i8s = 0.f;        // INT8: the scale of this thread's block (row, 32 columns) in the last QDQ'd state
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  const int64_t nchunks = (len + 63) / 64;
  auto issue_tma = [&](int64_t cj, int stg) {
    const uint32_t base = sbase + (uint32_t)stg * kStageBytes, bar = bar_tma0 + 8u * (uint32_t)stg;
    tc::mbar_expect_tx(bar, kStageBytes);
    const int tok = (int)(t0 + cj * 64);
    tc::tma_load_3d(base + ST_V, &tv, bar, slab * 64, h, tok);
    tc::tma_load_3d(base + ST_Q0, &tq, bar, 0, hq, tok);
    tc::tma_load_3d(base + ST_K0, &tk, bar, 0, hq, tok);
    tc::tma_load_3d(base + ST_Q1, &tq, bar, 64, hq, tok);
    tc::tma_load_3d(base + ST_K1, &tk, bar, 64, hq, tok);
  };
  if (tid == 0 && nchunks > 0) issue_tma(0, 0);
  int64_t tma_issued = nchunks > 0 ? 1 : 0;   // chunks whose TMA has been issued

  bool ok = true;
  bool aborted = false;
  // warp-uniform outcome: the TMEM loads that follow are warp-collective
  auto wait = [&](uint32_t bar, uint32_t par) { ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(bar, par)); };
  // warp 0 keeps the gates (g, beta) of the next chunk in registers: their loads overlap a chunk
  float nga = 0.f, ngb = 0.f, nba = 0.f, nbb = 0.f;
  auto load_gates = [&](int64_t cj) {
    const int64_t cc0 = cj * 64;
    const int Lj = (len - cc0) < 64 ? (int)(len - cc0) : 64;
    const int64_t base = (t0 + cc0) * p.Hv + h;
    nga = lt < Lj ? p.g[base + (int64_t)lt * p.Hv] : 0.f;
    ngb = lt + 32 < Lj ? p.g[base + (int64_t)(lt + 32) * p.Hv] : 0.f;
    nba = lt < Lj ? p.beta[base + (int64_t)lt * p.Hv] : 0.f;
    nbb = lt + 32 < Lj ? p.beta[base + (int64_t)(lt + 32) * p.Hv] : 0.f;
  };
  if (warp == 0 && nchunks > 0) load_gates(0);
  // warp 0: prefix sums of g inside chunk cj, Gam, decay to the chunk end, beta -> vecs[cj & 1]
  auto gates = [&](int64_t cj) {
    float* vg = vecs + (cj & 1) * 256;
    const int r0 = lt, r1 = lt + 32;
    float ga = nga, gb = ngb;
    const float ba = nba, bb = nbb;
    if (cj + 1 < nchunks) load_gates(cj + 1);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ya = __shfl_up_sync(0xffffffffu, ga, off);
      const float yb = __shfl_up_sync(0xffffffffu, gb, off);
      if (lt >= off) { ga += ya; gb += yb; }
    }
    gb += __shfl_sync(0xffffffffu, ga, 31);
    const float gl = __shfl_sync(0xffffffffu, gb, 31);
    vg[r0] = ga; vg[r1] = gb;
    vg[64 + r0] = __expf(ga); vg[64 + r1] = __expf(gb);
    vg[128 + r0] = __expf(gl - ga); vg[128 + r1] = __expf(gl - gb);
    vg[192 + r0] = ba; vg[192 + r1] = bb;
  };

  // wait for chunk cj's tiles, then issue its G1 = [Q; K] K^T and the TMA of chunk cj + 1
  auto start_chunk = [&](int64_t cj) {
    const int sj = (int)(cj & 1);
    wait(bar_tma0 + 8u * (uint32_t)sj, (uint32_t)((cj >> 1) & 1));
    if (__syncthreads_or(!ok)) return false;
    if (tid == 0) {
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t kb = ks >> 2, sub = (ks & 3) * 32;
        tc::mma_bf16(tmem + TM_G1, dadv(dStgK[sj], (kb ? ST_Q1 : ST_Q0) + sub),
                     dadv(dStgK[sj], (kb ? ST_K1 : ST_K0) + sub), IDESC_G1, ks > 0);
      }
      tc::mma_commit(bar_g1);
      if (cj + 1 < nchunks) issue_tma(cj + 1, sj ^ 1);
    }
    if (cj + 1 < nchunks) tma_issued = cj + 2;
    return true;
  };

  for (int64_t ci = 0; ci < nchunks; ++ci) {
    const int st = (int)(ci & 1);
    const int64_t c0 = ci * 64;
    const int L = (len - c0) < 64 ? (int)(len - c0) : 64;
    const uint32_t par = (uint32_t)(ci & 1);

    if (ci == 0) {
      if (!start_chunk(0)) { aborted = true; break; }
    }

    const float y_scale = s_scale;   // scale of this chunk's S0 operand (Y = Q S0); s_scale moves on below
    float* vgam = vecs + (ci & 1) * 256;   // this chunk's gate vectors
    float* vegam = vgam + 64;
    float* vdec = vgam + 128;
    float* vbeta = vgam + 192;
    if (ci == 0) {
      if (warp == 0) gates(0);
      __syncthreads();
    }
    // ---- A (rows of K K^T) and P (rows of Q K^T) from G1 ----
    wait(bar_g1, par);
    tc::tc_fence_after();
    if (ok) {
      float v[32];
      ld32(tmem, lane0, TM_G1 + col0, v);
      if (quad < 2) {   // G1 rows 0..63: Q K^T -> P (bf16 hi / lo, K-major [r][i])
        const int r = lane128;
        const float gr = vgam[r];
#pragma unroll
        for (int j = 0; j < 32; ++j) {   // the exponent is clamped so both select inputs are finite
          const int i = col0 + j;
          const float e = __expf(fminf(gr - vgam[i], 0.f)) * v[j];
          v[j] = i <= r ? e : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 hi, lo;
          split8(v + 8 * q, hi, lo);
          const uint32_t off = tc::sw128(r, 2 * (col0 + 8 * q));
          st16(sm, OFF_P + off, hi);
          st16(sm, OFF_P + 8 * KB + off, lo);
        }
      } else {          // G1 rows 64..127: K K^T -> A (fp32 rows)
        const int r = lane128 - 64;
        const float gr = vgam[r], br = vbeta[r];
        float4* dst = reinterpret_cast<float4*>(Am + r * A_LD + col0);
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float a4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = col0 + j + u;
            const float e = br * __expf(fminf(gr - vgam[i], 0.f)) * v[j + u];
            a4[u] = i < r ? e : 0.f;
          }
          dst[j >> 2] = make_float4(a4[0], a4[1], a4[2], a4[3]);
        }
      }
    }
    tc::tc_fence_before();
    if (__syncthreads_or(!ok)) { aborted = true; break; }

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution (into the T
    // buffer), then the off-diagonal blocks by levels of the block recurrence
    // T_ij = -T_ii sum_{j <= m < i} A_im T_mj  (level 1: i - j = 1, level 2: 2, level 3: 3)
    float* Tm = reinterpret_cast<float*>(sm + OFF_TT);   // fp32 [64][A_LD]; T''/T' overwrite it below
    {
      const int b0 = (tid >> 4) * 16, jj = tid & 15;
      if (tid < 64) {
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float* arow = Am + (b0 + r) * A_LD + b0;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;   // split accumulators: shorter chains
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
        // the blocks above the diagonal are zero
#pragma unroll
        for (int r = 0; r < 16; ++r)
#pragma unroll
          for (int bb = 1; bb < 4; ++bb)
            if (bb * 16 > b0) Tm[(b0 + r) * A_LD + bb * 16 + jj] = 0.f;
      }
      __syncthreads();
      // level tasks: one 1 x 4 tile (row rr, columns 4 c4 .. 4 c4 + 3) of a 16 x 16 block per thread
      const int blk = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
      // Y tile of block (bi, bj): sum_{m < 16 (bi - bj)} A[16 bi + rr][16 bj + m] T[16 bj + m][16 bj + c4 ..]
      auto ytile = [&](int bi, int bj, float* y) {
        y[0] = y[1] = y[2] = y[3] = 0.f;
#pragma unroll
        for (int m = 0; m < 16 * (bi - bj); ++m) {
          const float a = Am[(bi * 16 + rr) * A_LD + bj * 16 + m];
          const float4 t = *reinterpret_cast<const float4*>(Tm + (bj * 16 + m) * A_LD + bj * 16 + c4);
          y[0] = fmaf(a, t.x, y[0]); y[1] = fmaf(a, t.y, y[1]); y[2] = fmaf(a, t.z, y[2]); y[3] = fmaf(a, t.w, y[3]);
        }
      };
      // T tile of block (bi, bj) = -T_ii Y, Y a 16 x 16 scratch block
      auto ttile = [&](int bi, int bj, const float* Y) {
        float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float a = Tm[(bi * 16 + rr) * A_LD + bi * 16 + m];
          const float4 y = *reinterpret_cast<const float4*>(Y + m * 16 + c4);
          t4[0] = fmaf(a, y.x, t4[0]); t4[1] = fmaf(a, y.y, t4[1]); t4[2] = fmaf(a, y.z, t4[2]); t4[3] = fmaf(a, y.w, t4[3]);
        }
        *reinterpret_cast<float4*>(Tm + (bi * 16 + rr) * A_LD + bj * 16 + c4) = make_float4(-t4[0], -t4[1], -t4[2], -t4[3]);
      };
      auto put = [&](float* Y, const float* y) {
        *reinterpret_cast<float4*>(Y + rr * 16 + c4) = make_float4(y[0], y[1], y[2], y[3]);
      };
      float y[4];
      // level 1: blocks (1,0) (2,1) (3,2), 64 threads each
      if (blk < 3) { ytile(blk + 1, blk, y); put(scr + blk * 256, y); }
      __syncthreads();
      if (blk < 3) ttile(blk + 1, blk, scr + blk * 256);
      __syncthreads();
      // level 2: blocks (2,0) (3,1)
      if (blk < 2) { ytile(blk + 2, blk, y); put(scr + blk * 256, y); }
      __syncthreads();
      if (blk < 2) ttile(blk + 2, blk, scr + blk * 256);
      __syncthreads();
      // level 3: block (3,0)
      if (blk == 0) { ytile(3, 0, y); put(scr, y); }
      __syncthreads();
      if (blk == 0) ttile(3, 0, scr);
      __syncthreads();
    }
    // ---- T'' = T diag(beta), T' = T'' diag(Gam) as bf16 hi + lo, K-major [r][i] ----
    // (T is read into registers first: the outputs overwrite the T buffer)
    {
      float tv[2][8];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int task = tid + t * kThreads;   // 64 rows x 8 groups of 8 columns
        const int r = task >> 3, i0 = (task & 7) * 8;
        const float4 ta = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0);
        const float4 tb = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0 + 4);
        tv[t][0] = ta.x; tv[t][1] = ta.y; tv[t][2] = ta.z; tv[t][3] = ta.w;
        tv[t][4] = tb.x; tv[t][5] = tb.y; tv[t][6] = tb.z; tv[t][7] = tb.w;
      }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int task = tid + t * kThreads;
        const int r = task >> 3, i0 = (task & 7) * 8;
        const float4 ba = *reinterpret_cast<const float4*>(vbeta + i0);
        const float4 bb = *reinterpret_cast<const float4*>(vbeta + i0 + 4);
        const float4 ea = *reinterpret_cast<const float4*>(vegam + i0);
        const float4 eb = *reinterpret_cast<const float4*>(vegam + i0 + 4);
        const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
        const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
        float t2[8], t1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          t2[u] = tv[t][u] * bv[u];
          t1[u] = t2[u] * ev[u];
        }
        const uint32_t off = tc::sw128(r, 2 * i0);
        uint4 hi, lo;
        split8(t2, hi, lo);
        st16(sm, OFF_TT + off, hi);
        st16(sm, OFF_TT + 8 * KB + off, lo);
        split8(t1, hi, lo);
        st16(sm, OFF_TT + 16 * KB + off, hi);
        st16(sm, OFF_TT + 24 * KB + off, lo);
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      // U = T'' V: A = T'' (K-major), B = V (MN-major)
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_U, dadv(dTT, part * 8 * KB + ks * 32), dadv(dStgM[st], ST_V + ks * 2048), IDESC_U,
                       (part | ks) != 0);
      tc::mma_commit(bar_u);
      // W = T' K: A = T' (K-major), B = K (MN-major: the two 64-column blocks 16 KB apart)
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_W, dadv(dTT, 16 * KB + part * 8 * KB + ks * 32), dadv(dStgM[st], ST_K0 + ks * 2048),
                       IDESC_W, (part | ks) != 0);
      tc::mma_commit(bar_w);
    }

    // ---- W QDQ (one scale per chunk) -> W operand [r][c] for X ----
    wait(bar_w, par);
    tc::tc_fence_after();
    float sW = 1.f;
    {
      float w[64];   // row r = row64, columns [64 half, 64 half + 64)
      if (ok) {
        ld32(tmem, lane0, TM_W + half * 64, w);
        ld32(tmem, lane0, TM_W + half * 64 + 32, w + 32);
      }
      const bool act = lt < 16;
      const uint32_t abase = OFF_CW + (uint32_t)half * 8 * KB;
      if (p.w_qdq) {
        float m = 0.f;
        if (act) {
#pragma unroll
          for (int j = 0; j < 64; ++j) m = fmaxf(m, fabsf(w[j]));
        }
        m = warp_max(m);
        if (lt == 0) red[warp] = m;
        __syncthreads();
        float amax = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
        sW = qdq_scale(amax);
        const float rW = __frcp_rn(sW);
        if (act) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float c[8], d[8];
#pragma unroll
            for (int u = 0; u < 8; u += 2) qdq_pair(w[8 * q + u], w[8 * q + u + 1], rW, sW, c[u], c[u + 1], d[u], d[u + 1]);
            st16(sm, abase + tc::sw128(row64, 16 * q), pack8(c));
          }
        }
      } else if (act) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 hi, lo;
          split8(w + 8 * q, hi, lo);
          st16(sm, abase + tc::sw128(row64, 16 * q), hi);
          st16(sm, abase + 16 * KB + tc::sw128(row64, 16 * q), lo);
        }
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    if (__syncthreads_or(!ok)) { aborted = true; break; }
    if (tid == 0) {
      tc::tc_fence_after();
      // X = W S0 (M=64, N=64, K=128): (codes or W hi) x (S hi or codes) [+ W hi x S lo] [+ W lo x S hi]
      uint32_t aoff[3], boff[3];
      int np = 0;
      aoff[np] = 0; boff[np++] = 0;
      if (!s_exact) { aoff[np] = 0; boff[np++] = 16 * KB; }
      if (!p.w_qdq) { aoff[np] = 16 * KB; boff[np++] = 0; }
      for (int q = 0; q < np; ++q)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + TM_X, dadv(dCW, aoff[q] + (ks >> 2) * 8 * KB + (ks & 3) * 32), dadv(dS, boff[q] + ks * 2048),
                       IDESC_XY, (q | ks) != 0);
      tc::mma_commit(bar_x);
      // Y = Q S0: A = Q (the 64 Q rows of each 128-byte K block), B = S operand
      const int ny = s_exact ? 1 : 2;
      for (int q = 0; q < ny; ++q)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + TM_Y, dadv(dStgK[st], ((ks >> 2) ? ST_Q1 : ST_Q0) + (ks & 3) * 32),
                       dadv(dS, q * 16 * KB + ks * 2048), IDESC_XY, (q | ks) != 0);
      tc::mma_commit(bar_y);
    }

    // ---- Delta = U - W S0 -> Delta (bf16 hi/lo, for P Delta) and Dt = decay Delta (hi/lo), MN-major [i][j] ----
    wait(bar_u, par);
    wait(bar_x, par);
    tc::tc_fence_after();
    if (ok) {
      float xv[32], uv[32];
      ld32(tmem, lane0, TM_X + col0, xv);
      ld32(tmem, lane0, TM_U + col0, uv);
      if (lt < 16) {
        const int r = row64;
        const float f = sW * s_scale, dr = vdec[r];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float d[8], dt[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            d[u] = fmaf(-f, xv[8 * q + u], uv[8 * q + u]);
            dt[u] = dr * d[u];
          }
          const uint32_t off = tc::sw128(r, 2 * (col0 + 8 * q));
          uint4 hi, lo;
          split8(d, hi, lo);
          st16(sm, OFF_TT + off, hi);
          st16(sm, OFF_TT + 8 * KB + off, lo);
          split8(dt, hi, lo);
          st16(sm, OFF_TT + 16 * KB + off, hi);
          st16(sm, OFF_TT + 24 * KB + off, lo);
        }
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    if (__syncthreads_or(!ok)) { aborted = true; break; }
    if (tid == 0) {
      tc::tc_fence_after();
      // C = K^T Dt first: it is on the path to the next chunk: A = K^T (MN-major), B = Dt hi / lo (MN-major [i][j])
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_C, dadv(dStgM[st], ST_K0 + ks * 2048), dadv(dDl, 16 * KB + part * 8 * KB + ks * 2048),
                       IDESC_C, (part | ks) != 0);
      tc::mma_commit(bar_c);
      // P Delta = P_hi D_hi + P_hi D_lo + P_lo D_hi: A = P (K-major [r][i]), B = Delta (MN-major [i][j])
#pragma unroll
      for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_X, dadv(dP, (q == 2 ? 8 * KB : 0) + ks * 32), dadv(dDl, (q == 1 ? 8 * KB : 0) + ks * 2048),
                       IDESC_XY, (q | ks) != 0);
      tc::mma_commit(bar_pd);
    }

    // ---- S1 = Gam_L S0 + C, state QDQ at the 64-token boundary ----
    wait(bar_c, par);
    tc::tc_fence_after();
    {
      float s0[32], cv[32];
      if (ok) {
        ld32(tmem, lane0, TM_S + col0, s0);
        ld32(tmem, lane0, TM_C + col0, cv);
      }
      const float el = vegam[63];
#pragma unroll
      for (int j = 0; j < 32; ++j) s0[j] = fmaf(el, s0[j], cv[j]);
      const bool q = p.state_qdq == 1 && L == 64;
      if (q) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(s0[j]));
        m = warp_max(m);
        __syncthreads();   // red[] from the W QDQ is no longer read
        if (lt == 0) red[warp] = m;
        __syncthreads();
        float amax = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
        const float sS = qdq_scale(amax), rS = __frcp_rn(sS);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          float c[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2)
            qdq_pair(s0[8 * qq + u], s0[8 * qq + u + 1], rS, sS, c[u], c[u + 1], s0[8 * qq + u], s0[8 * qq + u + 1]);
          st16(sm, OFF_SHI + tc::sw128(lane128, 2 * (col0 + 8 * qq)), pack8(c));
        }
        s_exact = true;
        s_scale = sS;
      } else {
        if (p.state_qdq == 2 && L == 64) {   // INT8: this thread's 32 columns are one block of its row
          float m = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(s0[j]));
          const float sc = int8_scale(m), rc = __frcp_rn(sc);
#pragma unroll
          for (int j = 0; j < 32; ++j) s0[j] = int8_qdq_rcp(s0[j], rc, sc);
          i8s = sc;
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint4 hi, lo;
          split8(s0 + 8 * qq, hi, lo);
          const uint32_t off = tc::sw128(lane128, 2 * (col0 + 8 * qq));
          st16(sm, OFF_SHI + off, hi);
          st16(sm, OFF_SLO + off, lo);
        }
        s_exact = false;
        s_scale = 1.f;
      }
      if (ok) st32(tmem, lane0, TM_S + col0, s0);
      tc::tmem_st_wait();
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    if (__syncthreads_or(!ok)) { aborted = true; break; }
    tc::tc_fence_after();
    // the next chunk's G1 runs on the tensor cores while this chunk's outputs are written
    if (ci + 1 < nchunks && !start_chunk(ci + 1)) { aborted = true; break; }
    if (warp == 0 && ci + 1 < nchunks) gates(ci + 1);   // other buffer: this chunk's vectors stay intact
    // ---- outputs: o = scale (Gam Y + P Delta) for rows r < L ----
    wait(bar_y, par);
    wait(bar_pd, par);
    tc::tc_fence_after();
    if (ok) {
      float yv[32], pv[32];
      ld32(tmem, lane0, TM_Y + col0, yv);
      ld32(tmem, lane0, TM_X + col0, pv);
      if (lt < 16 && row64 < L) {
        const int r = row64;
        const float er = vegam[r] * y_scale;
        float4* out = reinterpret_cast<float4*>(p.o + ((t0 + c0 + r) * p.Hv + h) * (int64_t)p.dv + slab * 64 + col0);
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          out[j >> 2] = make_float4(p.scale * fmaf(er, yv[j], pv[j]), p.scale * fmaf(er, yv[j + 1], pv[j + 1]),
                                    p.scale * fmaf(er, yv[j + 2], pv[j + 2]), p.scale * fmaf(er, yv[j + 3], pv[j + 3]));
      }
    }

    __syncthreads();   // the next chunk's gate vectors are complete
  }

  if (!aborted && p.hT) {
    float s0[32];
    ld32(tmem, lane0, TM_S + col0, s0);
    float4* out = reinterpret_cast<float4*>(p.hT + sb + (int64_t)lane128 * p.dv + col0);
#pragma unroll
    for (int j = 0; j < 32; j += 4) out[j >> 2] = make_float4(s0[j], s0[j + 1], s0[j + 2], s0[j + 3]);
  }
  if (!aborted && p.sscale) {   // the final state was QDQ'd iff its last token was a 64th token
    const bool q = len > 0 && len % 64 == 0;
    const int64_t unit = (int64_t)n * p.Hv + h;
    if (p.state_qdq == 2)
      p.sscale[(unit * 128 + lane128) * (p.dv / kInt8BlockCols) + slab * 2 + half] = q ? i8s : 0.f;
    else if (tid == 0)
      p.sscale[unit * nslab + slab] = q ? s_scale : 0.f;
  }
  if (aborted) {
    if (tid == 0) atomicExch(p.status, 1);
    // the TMA of the last issued chunk may still be in flight: wait for it (bounded)
    const int64_t last = tma_issued - 1;
    if (last >= 0) tc::mbar_wait(bar_tma0 + 8u * (uint32_t)(last & 1), (uint32_t)((last >> 1) & 1), 1u << 16);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool chunk_tc_supported(const ChunkProblem& p) { return p.dk == 128 && !p.kda && p.dv % 64 == 0; }

cudaError_t launch_chunk_tc(const ChunkProblem& p, int* status, cudaStream_t stream) {
  const int64_t tokens = (int64_t)p.B * p.T;
  const int64_t blocks = (int64_t)p.N * p.Hv * (p.dv / 64);
  if (blocks == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv;
  // an empty batch still needs valid maps: point them at a one-token view (never loaded)
  const int64_t tmap = tokens > 0 ? tokens : 1;
  if (!make_bf16_map(&tq, p.q, 128, p.Hqk, tmap) || !make_bf16_map(&tk, p.k, 128, p.Hqk, tmap) ||
      !make_bf16_map(&tv, p.v, p.dv, p.Hv, tmap))
    return cudaErrorInvalidValue;
  TcParams tp{p.g, p.beta, p.h0, p.cu, p.o, p.hT, status, p.T, p.Hqk, p.Hv, p.dv, p.scale, p.state_qdq, p.w_qdq};
  tp.sscale = p.state_scales;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_tc_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(tq, tk, tv, tp);
  return cudaGetLastError();
}

}  // namespace gdn
