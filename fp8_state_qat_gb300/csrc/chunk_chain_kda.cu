// chunk_chain_kda.cu -- the state-carrying half of the chunked KDA forward (dk = 128) on the sm_103a
// tensor cores, after chunk_prep_kda.cu has staged every chunk's W^T, T'', P, the decayed Q / K and
// exp(gam_63) in the workspace.
//
// One CTA (256 threads) per (sequence n, v-head h, 64-column value slab); the slab is one state-QDQ
// tile, so its amax is CTA-local ("GDN state/W QAT foundation", "What does this PR do?"). With
// per-key-channel retention ("Add KDA prefill numerical emulation for QAT", "What does this PR
// do?") the chunk step is
//   X = W S0,  Delta = U - X,  U = T'' V
//   S1 = diag(exp(gam_63)) S0 + Kd^T Delta,  Kd = K o exp(gam_63 - gam);  QDQ(S1) at a 64-token boundary
//   o = scale (Qd S0 + P Delta),  Qd = Q o exp(gam)
// The state lives in TMEM as the accumulator of Kd^T Delta: the chain stores diag(exp(gam_63)) S0
// there and the MMAs add Kd_hi^T D_hi + Kd_hi^T D_lo + Kd_lo^T D_hi on top. S0 as an MMA operand
// (codes after a QDQ, else bf16 hi + lo) is double-buffered in shared memory, so Y = Qd S0 of one
// chunk never holds up the next state.
//
// Roles: the chain warpgroup (warps 4-7) runs X -> Delta -> C -> state epilogue, the only part that
// is serial from chunk to chunk; the output warpgroup (warps 0-3) issues Y, P Delta and the next U
// and writes o. The tensor pipe runs MMAs in issue order, so the output issuer places its MMAs
// behind the chain's: Y(c) after X(c) is issued (it runs while the chain computes Delta), P Delta
// and the next U after C(c) (they run while the chain updates the state). Each warpgroup issues
// from a thread on its own SM sub-partition. Every staged operand has one buffer, refilled once its
// last reader is done. Every wait is bounded; a warp whose wait gives up raises a CTA-wide abort
// flag, both warpgroups leave their loops together at their next checked barrier, TMA in flight
// is waited for (bounded), TMEM is freed.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace gdn {

cudaError_t launch_kda_prep(const ChunkProblem& p, const KdaLayout& lay, unsigned char* ws, cudaStream_t stream);

namespace {

constexpr int kThreads = 256;
constexpr int kOutIssuer = 64, kChainIssuer = 32;   // warp 2; warp 5 (index within the chain warpgroup)
constexpr uint32_t KB = 1024;
// shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_QD = 0;           // Qd hi (c < 64 | c >= 64), lo (same): [64 r][64 c] K-major blocks
constexpr uint32_t OFF_KD = 32 * KB;     // Kd hi | lo, same block layout (the MN-major A operand of C)
constexpr uint32_t OFF_TT = 64 * KB;     // T'' hi | lo [64 r][64 i] K-major
constexpr uint32_t OFF_V = 80 * KB;      // V slab [64 tok][64 j]
constexpr uint32_t OFF_WT = 88 * KB;     // W^T codes [128 c][64 r] (or hi | lo, 16 KB apart)
constexpr uint32_t OFF_S = 120 * KB;     // two S0 operand buffers [128 c][64 j] MN-major: codes or hi, lo at +16 KB
constexpr uint32_t OFF_DL = 184 * KB;    // Delta hi | lo ([i][j] MN-major, 8 KB each)
constexpr uint32_t OFF_P = 200 * KB;     // P hi | lo ([r][i] K-major)
constexpr uint32_t OFF_MISC = 216 * KB;  // S0 scale [4], S0-is-codes [4], partial maxima [4], flags
constexpr uint32_t kSmemBytes = OFF_MISC + 128 + 1024;

constexpr uint32_t TM_U = 0, TM_X = 64, TM_Y = 128, TM_S = 192, TM_PD = 256;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t IDESC_U = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);     // T'' (K) x V (MN)
constexpr uint32_t IDESC_X = tc::make_idesc(tc::kKindBF16, 64, 64, true, true);      // W^T (MN) x S0 (MN)
constexpr uint32_t IDESC_Y = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);     // Qd (K) x S0 (MN)
constexpr uint32_t IDESC_C = tc::make_idesc(tc::kKindBF16, 128, 64, true, true);     // Kd^T (MN) x Delta (MN)
constexpr uint32_t IDESC_PD = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);    // P (K) x Delta (MN)

enum : int {
  B_QD = 0, B_KD, B_TV, B_WC, B_PL, B_U, B_X, B_Y0, B_Y1, B_C, B_PD, B_SRDY0, B_SRDY1, B_DRDY, kNumBars
};

struct KdaChainParams {
  const int32_t* order;   // chain order of the sequences, or null (natural order)
  const float* vec;
  const float* h0;
  const int32_t* cu;
  const int32_t* lens;    // tokens run per sequence, or null (whole sequences)
  float* o;
  float* hT;
  int* status;
  int T, Hqk, Hv, dv;
  float scale;
  int state_qdq, w_qdq;
  float* sscale;   // final-state QDQ scales or null (layout: ChunkProblem::state_scales)
};

__device__ __forceinline__ void wg_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool wg_any(int id, bool pred) {   // warpgroup barrier that ORs pred
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, 128, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_chain_kda_kernel(const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap twt,
                       const __grid_constant__ CUtensorMap ttt, const __grid_constant__ CUtensorMap tpp,
                       const __grid_constant__ CUtensorMap tqd, const __grid_constant__ CUtensorMap tkd,
                       const KdaChainParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lt = tid & 31;
  const int quad = warp & 3;
  const uint32_t lane0 = (uint32_t)quad * 32u;
  const int lane128 = quad * 32 + lt;           // row of an M = 128 accumulator
  const int row64 = quad * 16 + (lt & 15);      // row of an M = 64 accumulator (16x32bx2 loads)
  const int half = lt >> 4;

  const int nslab = p.dv / 64;
  const int slab = blockIdx.x % nslab;
  const int h = (blockIdx.x / nslab) % p.Hv;
  const int n = p.order ? p.order[blockIdx.x / (nslab * p.Hv)] : (int)(blockIdx.x / (nslab * p.Hv));
  int64_t t0, len;
  if (p.cu) {
    t0 = p.cu[n];
    len = (int64_t)p.cu[n + 1] - t0;
  } else {
    t0 = (int64_t)n * p.T;
    len = p.T;
  }
  if (p.lens) len = p.lens[n];
  const int64_t nchunks = (len + 63) / 64;
  const int64_t slot0 = t0 / 64 + n;
  auto item = [&](int64_t cj) { return (slot0 + cj) * p.Hv + h; };
  auto chunk_len = [&](int64_t cj) { return (len - cj * 64) < 64 ? (int)(len - cj * 64) : 64; };

  float* const misc = reinterpret_cast<float*>(sm + OFF_MISC);
  float* const s_scale_slot = misc;                                   // [4], by chunk & 3
  int* const s_exact_slot = reinterpret_cast<int*>(misc + 4);         // [4]
  float* const red = misc + 8;                                        // [4]
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 12);
  volatile int* const x_issued = reinterpret_cast<volatile int*>(misc + 13);   // chunks whose X is issued
  volatile int* const c_issued = reinterpret_cast<volatile int*>(misc + 14);   // chunks whose C is issued
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) tc::mbar_init(bar(i), 1);
    *abort_flag = 0;
    *x_issued = 0;
    *c_issued = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tv);
    tc::tma_prefetch_desc(&twt);
    tc::tma_prefetch_desc(&ttt);
    tc::tma_prefetch_desc(&tpp);
    tc::tma_prefetch_desc(&tqd);
    tc::tma_prefetch_desc(&tkd);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  const uint64_t dQd = tc::make_sdesc(sbase + OFF_QD, 16, 1024);        // K-major Qd
  const uint64_t dKd = tc::make_sdesc(sbase + OFF_KD, 8 * KB, 1024);    // MN-major Kd^T (key blocks 8 KB apart)
  const uint64_t dTT = tc::make_sdesc(sbase + OFF_TT, 16, 1024);
  const uint64_t dV = tc::make_sdesc(sbase + OFF_V, 8 * KB, 1024);
  const uint64_t dWT = tc::make_sdesc(sbase + OFF_WT, 16 * KB, 1024);
  const uint64_t dS = tc::make_sdesc(sbase + OFF_S, 16 * KB, 1024);
  const uint64_t dD = tc::make_sdesc(sbase + OFF_DL, 8 * KB, 1024);     // Delta_hi, Delta_lo 8 KB apart
  const uint64_t dP = tc::make_sdesc(sbase + OFF_P, 16, 1024);

  auto tma_qd = [&](int64_t cj) {
    tc::mbar_expect_tx(bar(B_QD), 32 * KB);
    tc::tma_load_2d(sbase + OFF_QD, &tqd, bar(B_QD), 0, (int)(item(cj) * 256));
    tc::tma_load_2d(sbase + OFF_QD + 16 * KB, &tqd, bar(B_QD), 0, (int)(item(cj) * 256 + 128));
  };
  auto tma_kd = [&](int64_t cj) {
    tc::mbar_expect_tx(bar(B_KD), 32 * KB);
    tc::tma_load_2d(sbase + OFF_KD, &tkd, bar(B_KD), 0, (int)(item(cj) * 256));
    tc::tma_load_2d(sbase + OFF_KD + 16 * KB, &tkd, bar(B_KD), 0, (int)(item(cj) * 256 + 128));
  };
  auto tma_tv = [&](int64_t cj) {
    tc::mbar_expect_tx(bar(B_TV), 24 * KB);
    tc::tma_load_2d(sbase + OFF_TT, &ttt, bar(B_TV), 0, (int)(item(cj) * 128));
    tc::tma_load_3d(sbase + OFF_V, &tv, bar(B_TV), slab * 64, h, (int)(t0 + cj * 64));
  };
  auto tma_wc = [&](int64_t cj) {
    if (p.w_qdq) {
      tc::mbar_expect_tx(bar(B_WC), 16 * KB);
      tc::tma_load_2d(sbase + OFF_WT, &twt, bar(B_WC), 0, (int)(item(cj) * 128));
    } else {
      tc::mbar_expect_tx(bar(B_WC), 32 * KB);
      tc::tma_load_2d(sbase + OFF_WT, &twt, bar(B_WC), 0, (int)(item(cj) * 256));
      tc::tma_load_2d(sbase + OFF_WT + 16 * KB, &twt, bar(B_WC), 0, (int)(item(cj) * 256 + 128));
    }
  };
  auto tma_p = [&](int64_t cj) {
    tc::mbar_expect_tx(bar(B_PL), 16 * KB);
    tc::tma_load_2d(sbase + OFF_P, &tpp, bar(B_PL), 0, (int)(item(cj) * 128));
  };
  if (tid == 0 && nchunks > 0) {
    tma_qd(0);
    tma_kd(0);
    tma_tv(0);
    tma_wc(0);
    tma_p(0);
  }

  bool ok = true;
  auto live = [&]() { return ok && !*abort_flag; };
  auto wait = [&](int b, uint32_t par) {   // warp-collective; the decision to wait is warp-uniform
    if (__all_sync(0xffffffffu, live())) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(b), par));
      if (!ok && lt == 0) *abort_flag = 1;
    } else {
      ok = false;
    }
  };
  // warp-collective bounded wait until a chunk counter of the other warpgroup reaches `target`
  auto wait_count = [&](volatile int* ctr, int target) {
    if (__all_sync(0xffffffffu, live())) {
      bool reached = false;
      for (uint32_t it = 0; it < (1u << 22) && !reached; ++it) {
        reached = __all_sync(0xffffffffu, *ctr >= target);
        if (!reached && (it & 1023u) == 1023u && *abort_flag) break;
      }
      ok = reached;
      if (!ok && lt == 0) *abort_flag = 1;
    } else {
      ok = false;
    }
  };

  if (warp < 4) {
    // ================================ output warpgroup ================================
    auto issue_u = [&]() {   // U = T''_hi V + T''_lo V
      tc::tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_U, dadv(dTT, part * 8 * KB + ks * 32), dadv(dV, ks * 2048), IDESC_U, (part | ks) != 0);
      tc::mma_commit(bar(B_U));
    };
    // Only the issuing warp waits on the barriers that gate an issue or a refill: a refill of a
    // buffer follows its reader's completion, which follows that warp's wait on the fill, and
    // S0-ready / Y alternate between two barriers by chunk parity, so no barrier can run a phase
    // ahead of a warp still waiting on it. Every warp waits on Y and P Delta, whose accumulators
    // it reads.
    const bool issuer_warp = warp == kOutIssuer / 32;
    if (nchunks > 0 && issuer_warp) {
      wait(B_TV, 0);
      if (tid == kOutIssuer && live()) issue_u();
    }
    for (int64_t c = 0; c < nchunks; ++c) {
      const int L = chunk_len(c);
      const uint32_t par = (uint32_t)(c & 1), par2 = (uint32_t)((c >> 1) & 1);
      if (issuer_warp) {
        // T'' / V are free once U has read them
        wait(B_U, par);
        if (tid == kOutIssuer && c + 1 < nchunks && live()) tma_tv(c + 1);
        // ---- Y = Qd S0 once S0 is stored and X(c) is ahead of it in the tensor pipe ----
        wait(par ? B_SRDY1 : B_SRDY0, par2);
        wait(B_QD, par);
        wait_count(x_issued, (int)c + 1);
      }
      if (tid == kOutIssuer && live()) {
        const bool s_exact = s_exact_slot[c & 3] != 0;
        const uint32_t sb = par * 32 * KB;
        tc::tc_fence_after();
        // Qd_hi x S (codes or hi) + Qd_lo x S [+ Qd_hi x S_lo]; the two 64-column key blocks of Qd
        // are 8 KB apart, each 16-key step of S is 2 KB
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          if (q == 2 && s_exact) break;
          const uint32_t aoff = q == 1 ? 16 * KB : 0, boff = sb + (q == 2 ? 16 * KB : 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + TM_Y, dadv(dQd, aoff + (ks >> 2) * 8 * KB + (ks & 3) * 32), dadv(dS, boff + ks * 2048),
                         IDESC_Y, (q | ks) != 0);
        }
        tc::mma_commit(bar(par ? B_Y1 : B_Y0));
      }
      // ---- P Delta = P_hi D_hi + P_hi D_lo + P_lo D_hi and the next U, behind C(c) ----
      if (issuer_warp) {
        wait(B_DRDY, par);
        wait(B_PL, par);
        wait_count(c_issued, (int)c + 1);
      }
      if (tid == kOutIssuer && live()) {
        tc::tc_fence_after();
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16(tmem + TM_PD, dadv(dP, (q == 2 ? 8 * KB : 0) + ks * 32), dadv(dD, (q == 1 ? 8 * KB : 0) + ks * 2048),
                         IDESC_PD, (q | ks) != 0);
        tc::mma_commit(bar(B_PD));
      }
      if (c + 1 < nchunks && issuer_warp) {   // the chain stored Delta, so it has read U
        wait(B_TV, par ^ 1u);
        if (tid == kOutIssuer && live()) issue_u();
      }
      // ---- refills once their readers are done: Qd after Y, P after P Delta ----
      wait(par ? B_Y1 : B_Y0, par2);
      if (tid == kOutIssuer && c + 1 < nchunks && live()) tma_qd(c + 1);
      wait(B_PD, par);
      if (tid == kOutIssuer && c + 1 < nchunks && live()) tma_p(c + 1);
      // ---- o = scale (Y + P Delta), rows r < L; the scale slot is rewritten only after Y(c + 2) ----
      tc::tc_fence_after();
      {
        const float y_scale = s_scale_slot[c & 3];
        float yv[32], pv[32];
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_Y), yv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_Y + 16), yv + 16);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_PD), pv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_PD + 16), pv + 16);
        tc::tmem_ld_wait();
        if (row64 < L) {
          float4* out = reinterpret_cast<float4*>(p.o + ((t0 + c * 64 + row64) * p.Hv + h) * (int64_t)p.dv +
                                                  slab * 64 + half * 32);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            out[j >> 2] = make_float4(p.scale * fmaf(y_scale, yv[j], pv[j]), p.scale * fmaf(y_scale, yv[j + 1], pv[j + 1]),
                                      p.scale * fmaf(y_scale, yv[j + 2], pv[j + 2]), p.scale * fmaf(y_scale, yv[j + 3], pv[j + 3]));
        }
      }
      tc::tc_fence_before();
      if (wg_any(1, !live())) break;
    }
  } else {
    // ================================ chain warpgroup ================================
    const int ctid = tid - 128;
    const bool issuer_warp = warp == 4 + kChainIssuer / 32;
    const int64_t sbg = ((int64_t)n * p.Hv + h) * 128 * p.dv + slab * 64;   // S[c][j] at sbg + c dv + j
    // the W scale of the current chunk (read from global one chunk ahead)
    float sw_next = 1.f;
    {   // S0: operand buffer 0 (bf16 hi + lo) and diag(exp(gam_63)) S0 into the TMEM state
      float s0[64];
      if (p.h0) {
        const float4* src = reinterpret_cast<const float4*>(p.h0 + sbg + (int64_t)lane128 * p.dv);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 f = src[j];
          s0[4 * j] = f.x; s0[4 * j + 1] = f.y; s0[4 * j + 2] = f.z; s0[4 * j + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) s0[j] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint4 h16, l16;
        split8(s0 + 8 * q, h16, l16);
        const uint32_t off = tc::sw128(lane128, 16 * q);
        st16(sm, OFF_S + off, h16);
        st16(sm, OFF_S + 16 * KB + off, l16);
      }
      if (nchunks > 0) {
        const float el0 = p.vec[item(0) * 256 + lane128];
        sw_next = p.vec[item(0) * 256 + 192];
#pragma unroll
        for (int j = 0; j < 64; ++j) s0[j] *= el0;
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::tmem_st16(tc::tmem_addr(tmem, lane0, TM_S + 16 * q), s0 + 16 * q);
        tc::tmem_st_wait();
      } else if (p.hT) {   // an empty sequence: hT = h0
        float4* out = reinterpret_cast<float4*>(p.hT + sbg + (int64_t)lane128 * p.dv);
#pragma unroll
        for (int j = 0; j < 64; j += 4) out[j >> 2] = make_float4(s0[j], s0[j + 1], s0[j + 2], s0[j + 3]);
      }
    }
    if (ctid == 0) {
      s_scale_slot[0] = 1.f;
      s_exact_slot[0] = 0;
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    wg_sync(2);
    if (ctid == 0) tc::mbar_arrive(bar(B_SRDY0));
    bool s_exact = false;
    float s_scale = 1.f;
    float i8s[2] = {0.f, 0.f};   // INT8: this row's two block scales of the last QDQ'd state
    for (int64_t c = 0; c < nchunks; ++c) {
      const int L = chunk_len(c);
      const uint32_t par = (uint32_t)(c & 1);
      const uint32_t sb = par * 32 * KB;          // this chunk's S0 operand buffer
      const float f = sw_next * s_scale;          // X holds codes x codes: W scale x S0 scale
      const float el1 = (c + 1 < nchunks) ? p.vec[item(c + 1) * 256 + lane128] : 1.f;   // the next chunk's decay
      if (c + 1 < nchunks) sw_next = p.vec[item(c + 1) * 256 + 192];
      // ---- X = W S0 ----
      if (issuer_warp) wait(B_WC, par);
      if (ctid == kChainIssuer && live()) {
        tc::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + TM_X, dadv(dWT, ks * 2048), dadv(dS, sb + ks * 2048), IDESC_X, ks > 0);
        if (!s_exact) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + TM_X, dadv(dWT, ks * 2048), dadv(dS, sb + 16 * KB + ks * 2048), IDESC_X, 1);
        }
        if (!p.w_qdq) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + TM_X, dadv(dWT, 16 * KB + ks * 2048), dadv(dS, sb + ks * 2048), IDESC_X, 1);
        }
        tc::mma_commit(bar(B_X));
        *x_issued = (int)c + 1;
      }
      wait(B_X, par);
      if (ctid == kChainIssuer && c + 1 < nchunks && live()) tma_wc(c + 1);
      // ---- Delta = U - f X -> hi | lo ----
      wait(B_U, par);
      if (c > 0) wait(B_PD, (uint32_t)((c - 1) & 1));   // the previous P Delta has read Delta
      tc::tc_fence_after();
      {
        float xv[32], uv[32];
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_X), xv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_X + 16), xv + 16);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_U), uv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_U + 16), uv + 16);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float d[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) d[u] = fmaf(-f, xv[8 * q + u], uv[8 * q + u]);
          uint4 h16, l16;
          split8(d, h16, l16);
          const uint32_t off = tc::sw128(row64, 2 * (half * 32 + 8 * q));
          st16(sm, OFF_DL + off, h16);
          st16(sm, OFF_DL + 8 * KB + off, l16);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      if (wg_any(2, !live())) break;
      if (ctid == 0) tc::mbar_arrive(bar(B_DRDY));   // Delta stored; U and X read
      // ---- state += Kd_hi^T D_hi + Kd_hi^T D_lo + Kd_lo^T D_hi ----
      if (issuer_warp) wait(B_KD, par);
      if (ctid == kChainIssuer && live()) {
        tc::tc_fence_after();
#pragma unroll
        for (int q = 0; q < 3; ++q)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16(tmem + TM_S, dadv(dKd, (q == 2 ? 16 * KB : 0) + ks * 2048), dadv(dD, (q == 1 ? 8 * KB : 0) + ks * 2048),
                         IDESC_C, 1);
        tc::mma_commit(bar(B_C));
        *c_issued = (int)c + 1;
      }
      wait(B_C, par);
      if (ctid == kChainIssuer && c + 1 < nchunks && live()) tma_kd(c + 1);   // Kd is free once C has read it
      // ---- S1 from TMEM; QDQ at the 64-token boundary; into the other operand buffer once
      // Y(c - 1) has read it; diag(exp(gam_63)) S1 back into TMEM for the next chunk ----
      tc::tc_fence_after();
      float s1[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::tmem_ld16(tc::tmem_addr(tmem, lane0, TM_S + 16 * q), s1 + 16 * q);
      tc::tmem_ld_wait();
      const uint32_t nb = (par ^ 1u) * 32 * KB;
      if (c > 0) wait(par ? B_Y0 : B_Y1, (uint32_t)(((c - 1) >> 1) & 1));
      if (p.state_qdq == 1 && L == 64) {
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = fabsf(s1[u]);
#pragma unroll
        for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], fabsf(s1[j]));
        const float mm = warp_absmax(fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                           fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))));
        if (lt == 0) red[quad] = mm;
        wg_sync(2);
        const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        const float sS = qdq_scale(amax), rS = __frcp_rn(sS);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float cd[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2)
            qdq_pair(s1[8 * q + u], s1[8 * q + u + 1], rS, sS, cd[u], cd[u + 1], s1[8 * q + u], s1[8 * q + u + 1]);
          st16(sm, OFF_S + nb + tc::sw128(lane128, 16 * q), pack8(cd));
        }
        s_exact = true;
        s_scale = sS;
      } else {
        if (p.state_qdq == 2 && L == 64) {   // INT8: this row's two 32-column blocks, in registers
#pragma unroll
          for (int b0 = 0; b0 < 64; b0 += kInt8BlockCols) {
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < kInt8BlockCols; ++j) m = fmaxf(m, fabsf(s1[b0 + j]));
            const float sc = int8_scale(m), rc = __frcp_rn(sc);
#pragma unroll
            for (int j = 0; j < kInt8BlockCols; ++j) s1[b0 + j] = int8_qdq_rcp(s1[b0 + j], rc, sc);
            i8s[b0 / kInt8BlockCols] = sc;
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 h16, l16;
          split8(s1 + 8 * q, h16, l16);
          const uint32_t off = tc::sw128(lane128, 16 * q);
          st16(sm, OFF_S + nb + off, h16);
          st16(sm, OFF_S + nb + 16 * KB + off, l16);
        }
        s_exact = false;
        s_scale = 1.f;
      }
      if (c + 1 < nchunks) {
        float e[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int u = 0; u < 16; ++u) e[u] = el1 * s1[16 * q + u];
          tc::tmem_st16(tc::tmem_addr(tmem, lane0, TM_S + 16 * q), e);
        }
        tc::tmem_st_wait();
      } else if (live() && p.hT) {
        float4* out = reinterpret_cast<float4*>(p.hT + sbg + (int64_t)lane128 * p.dv);
#pragma unroll
        for (int j = 0; j < 64; j += 4) out[j >> 2] = make_float4(s1[j], s1[j + 1], s1[j + 2], s1[j + 3]);
      }
      if (ctid == 0) {
        s_scale_slot[(c + 1) & 3] = s_scale;
        s_exact_slot[(c + 1) & 3] = s_exact ? 1 : 0;
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      if (wg_any(2, !live())) break;
      if (ctid == 0) tc::mbar_arrive(bar(par ? B_SRDY0 : B_SRDY1));   // S0 of chunk c + 1 is stored
    }
    if (live() && p.sscale) {   // the final state was QDQ'd iff its last token was a 64th token
      const bool q = len > 0 && len % 64 == 0;
      const int64_t unit = (int64_t)n * p.Hv + h;
      if (p.state_qdq == 2) {
        float* dst = p.sscale + (unit * 128 + lane128) * (p.dv / kInt8BlockCols) + slab * 2;
        dst[0] = q ? i8s[0] : 0.f;
        dst[1] = q ? i8s[1] : 0.f;
      } else if (ctid == 0) {
        p.sscale[unit * nslab + slab] = q ? s_scale : 0.f;
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) {
      atomicExch(p.status, 1);
      const int tx_bars[5] = {B_QD, B_KD, B_TV, B_WC, B_PL};
      for (int i = 0; i < 5; ++i) {   // TMA still landing: wait for each barrier's current phase, bounded
        tc::mbar_wait(bar(tx_bars[i]), 0, 1u << 14);
        tc::mbar_wait(bar(tx_bars[i]), 1, 1u << 14);
      }
    }
    __syncthreads();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool kda_split_supported(const ChunkProblem& p) {
  return p.dk == 128 && p.kda && p.dv % 64 == 0 && (reinterpret_cast<uintptr_t>(p.g) & 15) == 0;   // g read as float4
}

KdaLayout kda_split_layout(const ChunkProblem& p) {
  KdaLayout l{};
  const int64_t tokens = (int64_t)p.B * p.T;
  l.slots = tokens / 64 + p.N;
  l.items = l.slots * p.Hv;
  l.wt_item_bytes = p.w_qdq ? 16 * KB : 32 * KB;
  auto up = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
  l.off_wt = up(kStatusBytes);
  l.off_tt = up(l.off_wt + (size_t)l.items * l.wt_item_bytes);
  l.off_p = up(l.off_tt + (size_t)l.items * 16 * KB);
  l.off_qd = up(l.off_p + (size_t)l.items * 16 * KB);
  l.off_kd = up(l.off_qd + (size_t)l.items * 32 * KB);
  l.off_vec = up(l.off_kd + (size_t)l.items * 32 * KB);
  l.off_order = up(l.off_vec + (size_t)l.items * 1024);
  l.total = l.off_order + (size_t)p.N * 4;
  return l;
}

cudaError_t launch_kda_split(const ChunkProblem& p, void* ws, cudaStream_t stream) {
  const KdaLayout lay = kda_split_layout(p);
  if (lay.items * 256 >= (int64_t)1 << 31) return cudaErrorInvalidValue;   // TMA row coordinates are int32
  unsigned char* w = static_cast<unsigned char*>(ws);
  cudaError_t e = launch_kda_prep(p, lay, w, stream);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.N * p.Hv * (p.dv / 64);
  if (blocks == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  CUtensorMap tv, twt, ttt, tpp, tqd, tkd;
  if (!make_bf16_map(&tv, p.v, p.dv, p.Hv, tokens > 0 ? tokens : 1) ||
      !make_bf16_rows_map(&twt, w + lay.off_wt, lay.items * (p.w_qdq ? 128 : 256), 128) ||
      !make_bf16_rows_map(&ttt, w + lay.off_tt, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tpp, w + lay.off_p, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tqd, w + lay.off_qd, lay.items * 256, 128) ||
      !make_bf16_rows_map(&tkd, w + lay.off_kd, lay.items * 256, 128))
    return cudaErrorInvalidValue;
  const int32_t* order = stage_chain_order(p, w, lay.off_order, stream, &e);
  if (e != cudaSuccess) return e;
  KdaChainParams cp{order, reinterpret_cast<const float*>(w + lay.off_vec), p.h0, p.cu, p.lens, p.o, p.hT,
                    reinterpret_cast<int*>(ws), p.T, p.Hqk, p.Hv, p.dv, p.scale, p.state_qdq, p.w_qdq};
  cp.sscale = p.state_scales;
  e = cudaFuncSetAttribute(chunk_chain_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_chain_kda_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(tv, twt, ttt, tpp, tqd, tkd, cp);
  return cudaGetLastError();
}

}  // namespace gdn
