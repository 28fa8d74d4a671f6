// chunk_chain.cu -- the state-carrying half of the chunked gated-delta-rule forward (dk = 128) on
// the sm_103a tensor cores, after chunk_prep.cu has staged every chunk's W, T'', P and gate
// vectors in the workspace.
//
// One CTA (256 threads) per (sequence n, v-head h, 64-column value slab); the slab is one
// state-QDQ tile (all 128 key rows x 64 value columns), so its amax is CTA-local ("GDN state/W QAT
// foundation", "What does this PR do?"); with the INT8 codec each thread's key row holds its two
// 32-column blocks, and the QDQ'd state is carried as bf16 hi + lo. Two warpgroups split each chunk:
//   chain  (warps 4-7)  [X; Y] = [W; Q] S0 -> Delta = U - X, Dt = exp(gam_63 - gam) Delta ->
//                       C = K^T Dt -> S1 = Gam_63 S0 + C, QDQ(S1) at a 64-token boundary -> the
//                       next chunk. Only this loop is serial from chunk to chunk. X and Y come
//                       from one M = 128 product whose A rows interleave W and Q in 16-row groups,
//                       so X lands in TMEM lanes 0-15 and Y in lanes 16-31 of each quadrant (the
//                       M = 64 row layout) and Y costs no separate MMA or wait. It also refills
//                       the stages (W, Q, K, gate vectors) once their last readers are done.
//   output (warps 0-3)  U = T'' V, P Delta (P staged by the prep), o = scale (Gam Y + P Delta)
//                       through a shared-memory tile and one TMA store per chunk; U of the next
//                       chunk is issued right after P Delta, ahead of the chain's next [X; Y].
//                       Its warps also issue every TMA copy of the CTA (stage refills once the
//                       chain signals a stage free, T'' / V, P, the o store), so that neither MMA
//                       issuer issues anything but MMAs.
// The state S0 (fp32) lives in the chain's registers (one key row of the slab per thread) and, as
// the MMA operand, in shared memory as bf16 hi + lo, or as exact E4M3 codes once QDQ'd (the scale
// is applied in the epilogues). W arrives as codes (exact in bf16) with W QDQ, else as bf16 hi +
// lo (the lo part as a separate M = 64 product accumulating onto X); T'' and P as hi + lo; Delta
// and Dt are split into hi + lo before their MMAs.
//
// Hand-offs are mbarriers (TMA transactions, MMA commits, and one-arrival signals: "U consumed",
// "Delta stored" and "stage free" from the chain, "Y read" from the output warpgroup). Every wait is bounded; a
// warp whose wait gives up raises a CTA-wide abort flag, both warpgroups leave their loops at
// their next checked barrier, TMA in flight is waited for (bounded), TMEM is freed.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace gdn {

cudaError_t launch_chunk_prep(const ChunkProblem& p, const SplitLayout& lay, unsigned char* ws, cudaStream_t stream);

namespace {

constexpr int kThreads = 256;
// The threads that issue each warpgroup's MMAs and TMA loads. A tcgen05.mma issues slowly while other
// warps on the same SM sub-partition (warp id mod 4) keep its FP32 pipes busy, so the two issuers
// sit on different sub-partitions.
#ifndef GDN_OUT_ISSUER
#define GDN_OUT_ISSUER 64     // warp 2
#endif
#ifndef GDN_CHAIN_ISSUER
#define GDN_CHAIN_ISSUER 32   // warp 5 (index within the chain warpgroup)
#endif
constexpr int kOutIssuer = GDN_OUT_ISSUER, kChainIssuer = GDN_CHAIN_ISSUER;
constexpr uint32_t KB = 1024;
// shared memory map (byte offsets from a 1024-byte aligned base)
//   stage s (two, by chunk parity) at s * kStage: A0 | A1 (16 KB each: key columns 0-63 | 64-127 of
//   the [W; Q] operand, 128 rows; rows 32 g .. 32 g + 15 are W rows 16 g .. 16 g + 15, rows 32 g +
//   16 .. 32 g + 31 the Q rows 16 g .. 16 g + 15), then K0 | K1 (8 KB each, [64 tok][64])
constexpr uint32_t kStage = 50 * KB;
constexpr uint32_t SA0 = 0, SK0 = 32 * KB;
constexpr uint32_t OFF_VEC = 100 * KB;  // gate vectors of chunk c in slot c mod 4 (1 KB each)
constexpr uint32_t OFF_WLO = 104 * KB;  // W lo without W QDQ: key block 0 | 1, [64 r][64 c] K-major
constexpr uint32_t OFF_TT = 120 * KB;   // T'' hi | lo rows interleaved, [128][64 i] K-major
constexpr uint32_t OFF_V = 136 * KB;    // V slab [64 tok][64 j]
constexpr uint32_t OFF_SHI = 144 * KB;  // S0 operand [128 c][64 j] MN-major; lo at +16 KB
constexpr uint32_t OFF_DL = 176 * KB;   // Delta hi, lo, Dt hi, lo ([i][j] MN-major, 8 KB each)
constexpr uint32_t OFF_PO = 208 * KB;   // P hi | lo rows interleaved ([128][i] K-major); once P Delta is done, the o tile
                                        // (two [64 tok][32 j] fp32 halves, 128-byte swizzled rows)
constexpr uint32_t OFF_MISC = 224 * KB; // S0 scales [4] by chunk mod 4, partial maxima [4], abort flag
constexpr uint32_t kSmemBytes = OFF_MISC + 64 + 1024;   // + slack to align the base
static_assert(kSmemBytes <= 227 * KB, "shared memory map exceeds the per-CTA limit");

// TMEM columns. M = 128 products whose A rows interleave two 64-row matrices in 16-row groups put
// the first one's result in lanes 0-15 and the second's in lanes 16-31 of each quadrant (the M = 64
// row layout, row 16 q + i in lane 32 q + i):
//   [X; Y] of chunk c   TM_XY + 64 (c & 1)   [W; Q] S0
//   U                   TM_U                 [T''_hi; T''_lo] V         (U = the two halves summed)
//   C                   TM_C (128 columns)   K^T [Dt_hi | Dt_lo]        (C = left + right)
//   P Delta             TM_PD (128 columns)  [P_hi; P_lo] [D_hi | D_lo] (P Delta = the four parts summed)
constexpr uint32_t TM_XY = 0, TM_U = 128, TM_C = 192, TM_PD = 320;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t IDESC_U = tc::make_idesc(tc::kKindBF16, 128, 64, false, true);    // [T''hi; T''lo] (K) x V (MN)
constexpr uint32_t IDESC_XY = tc::make_idesc(tc::kKindBF16, 128, 64, false, true);   // [W; Q] (K) x S0 (MN)
constexpr uint32_t IDESC_WLO = tc::make_idesc(tc::kKindBF16, 64, 64, false, true);   // W lo (K) x S0 (MN)
constexpr uint32_t IDESC_C = tc::make_idesc(tc::kKindBF16, 128, 128, true, true);    // K^T (MN) x [Dt hi | lo] (MN)
constexpr uint32_t IDESC_PD = tc::make_idesc(tc::kKindBF16, 128, 128, false, true);  // [P hi; lo] (K) x [D hi | lo] (MN)

enum : int {
  B_QK0 = 0, B_QK1, B_TV, B_P, B_WLO, B_U, B_XY0, B_XY1, B_C, B_PD, B_DRDY, B_OD0, B_OD1, B_SF0, B_SF1, kNumBars
};
// Threads that issue TMA copies. The MMA issuers issue nothing else: a thread's tcgen05.mma queues
// behind the bulk copies it issued before, so refills from an issuer sit on the chain's path.
constexpr int kTvLoader = 32;     // warp 1: T'' / V
constexpr int kStageLoader = 96;  // warp 3: stage refills, the o store and P

struct ChainParams {
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
// barrier over one warpgroup (named barrier `id`) that also ORs `pred` across its 128 threads
__device__ __forceinline__ bool wg_any(int id, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, 128, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap tq16, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tw16,
                   const __grid_constant__ CUtensorMap tw64, const __grid_constant__ CUtensorMap ttt,
                   const __grid_constant__ CUtensorMap tpp, const __grid_constant__ CUtensorMap tout,
                   const ChainParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lt = tid & 31;
  const int quad = warp & 3;
  const uint32_t lane0 = (uint32_t)quad * 32u;
  const int lane128 = quad * 32 + lt;           // row of an M = 128 accumulator (32x32b loads)
  const int row64 = quad * 16 + (lt & 15);      // row of an M = 64 accumulator (16x32bx2 loads)
  const int half = lt >> 4;                     // ... and its column half: [32 half, 32 half + 32)

  const int nslab = p.dv / 64;
  const int slab = blockIdx.x % nslab;
  const int h = (blockIdx.x / nslab) % p.Hv;
  const int n = p.order ? p.order[blockIdx.x / (nslab * p.Hv)] : (int)(blockIdx.x / (nslab * p.Hv));
  const int hq = h / (p.Hv / p.Hqk);
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
  const int64_t slot0 = t0 / 64 + n;   // workspace slot of chunk 0
  auto item = [&](int64_t cj) { return (slot0 + cj) * p.Hv + h; };
  auto chunk_len = [&](int64_t cj) { return (len - cj * 64) < 64 ? (int)(len - cj * 64) : 64; };
  auto vecs = [&](int64_t cj) { return reinterpret_cast<const float*>(sm + OFF_VEC + (uint32_t)(cj & 3) * KB); };

  float* const misc = reinterpret_cast<float*>(sm + OFF_MISC);
  float* const s_scale_slot = misc;                                       // [4], by chunk mod 4
  float* const red = misc + 4;                                            // [4]
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 8);
  auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) tc::mbar_init(bar(i), 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tq16);
    tc::tma_prefetch_desc(&tk);
    tc::tma_prefetch_desc(&tv);
    tc::tma_prefetch_desc(&tw16);
    tc::tma_prefetch_desc(&tw64);
    tc::tma_prefetch_desc(&ttt);
    tc::tma_prefetch_desc(&tpp);
    tc::tma_prefetch_desc(&tout);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // operand descriptors (128-byte swizzle, 8-row groups 1024 bytes apart)
  const uint64_t dStgA = tc::make_sdesc(sbase + SA0, 16, 1024);       // K-major [W; Q] of stage 0
  const uint64_t dStgM = tc::make_sdesc(sbase + SK0, 8 * KB, 1024);   // MN-major K^T of stage 0
  const uint64_t dWlo = tc::make_sdesc(sbase + OFF_WLO, 16, 1024);
  const uint64_t dTT = tc::make_sdesc(sbase + OFF_TT, 16, 1024);
  const uint64_t dV = tc::make_sdesc(sbase + OFF_V, 8 * KB, 1024);
  const uint64_t dS = tc::make_sdesc(sbase + OFF_SHI, 16 * KB, 1024);
  const uint64_t dDl = tc::make_sdesc(sbase + OFF_DL, 8 * KB, 1024);   // [D hi | D lo], then [Dt hi | Dt lo] at +16 KB
  const uint64_t dP = tc::make_sdesc(sbase + OFF_PO, 16, 1024);

  const int64_t wrows = p.w_qdq ? 128 : 256;   // staged W rows per item: codes, or hi then lo
  auto tma_qk = [&](int64_t cj) {   // [W; Q], K tiles and gate vectors of chunk cj into stage cj & 1
    const int s = (int)(cj & 1);
    const uint32_t base = sbase + (uint32_t)s * kStage, b = bar(B_QK0 + s);
    tc::mbar_expect_tx(b, 48 * KB + 1024);
    const int tok = (int)(t0 + cj * 64);
    const int wr = (int)(item(cj) * wrows);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t dst = base + SA0 + (uint32_t)kb * 16 * KB + (uint32_t)g * 4 * KB;
        tc::tma_load_2d(dst, &tw16, b, 0, wr + kb * 64 + 16 * g);
        tc::tma_load_3d(dst + 2 * KB, &tq16, b, kb * 64, hq, tok + 16 * g);
      }
    tc::tma_load_3d(base + SK0, &tk, b, 0, hq, tok);
    tc::tma_load_3d(base + SK0 + 8 * KB, &tk, b, 64, hq, tok);
    tc::bulk_load(sbase + OFF_VEC + (uint32_t)(cj & 3) * KB, p.vec + item(cj) * 256, 1024, b);
  };
  auto tma_wlo = [&](int64_t cj) {  // W lo (without W QDQ) of chunk cj
    tc::mbar_expect_tx(bar(B_WLO), 16 * KB);
    tc::tma_load_2d(sbase + OFF_WLO, &tw64, bar(B_WLO), 0, (int)(item(cj) * 256 + 128));
    tc::tma_load_2d(sbase + OFF_WLO + 8 * KB, &tw64, bar(B_WLO), 0, (int)(item(cj) * 256 + 192));
  };
  auto tma_tv = [&](int64_t cj) {   // T'' hi | lo and the V slab of chunk cj
    tc::mbar_expect_tx(bar(B_TV), 24 * KB);
    tc::tma_load_2d(sbase + OFF_TT, &ttt, bar(B_TV), 0, (int)(item(cj) * 128));
    tc::tma_load_3d(sbase + OFF_V, &tv, bar(B_TV), slab * 64, h, (int)(t0 + cj * 64));
  };
  auto tma_p = [&](int64_t cj) {    // P hi | lo of chunk cj
    tc::mbar_expect_tx(bar(B_P), 16 * KB);
    tc::tma_load_2d(sbase + OFF_PO, &tpp, bar(B_P), 0, (int)(item(cj) * 128));
  };
  // launched as a programmatic dependent of the prep kernel: everything above overlaps its last
  // wave; its staging is read only after it has completed (a no-op without that launch attribute)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && nchunks > 0) {
    tma_qk(0);
    tma_tv(0);
    tma_p(0);
    if (!p.w_qdq) tma_wlo(0);
    if (nchunks > 1) tma_qk(1);
  }

  // Bounded waits never leave the loops on their own: a warp whose wait gives up clears `ok`
  // and raises the abort flag; all warps of its group still reach the group's next checked
  // barrier (wg_any), where they stop together. Nothing is issued once live() is false.
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

  if (warp < 4) {
    // ================================ output warpgroup ================================
    auto issue_u = [&]() {   // [T''_hi; T''_lo] V
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        tc::mma_bf16(tmem + TM_U, dadv(dTT, ks * 32), dadv(dV, ks * 2048), IDESC_U, ks != 0);
      tc::mma_commit(bar(B_U));
    };
    if (nchunks > 0) {
      wait(B_TV, 0);
      if (tid == kOutIssuer && live()) issue_u();
    }
    for (int64_t c = 0; c < nchunks; ++c) {
      const int s = (int)(c & 1);
      const int L = chunk_len(c);
      const uint32_t par = (uint32_t)(c & 1);
      // T'' / V are free once U has completed: fetch the next chunk's, a whole chunk ahead
      if (warp == kTvLoader / 32) {
        wait(B_U, par);
        if (tid == kTvLoader && c + 1 < nchunks && live()) tma_tv(c + 1);
      }
      // ---- P Delta and the next U, once the chain's C has completed: they run in the tensor pipe
      // while the chain carries out its state epilogue, never next to its [X; Y] or C ----
      wait(B_DRDY, par);
      // S0's scale and the row's Gam: written / landed before the chain stored Delta
      const float y_scale = s_scale_slot[c & 3];
      const float egam_r = vecs(c)[64 + row64];
      wait(B_SF0 + s, (uint32_t)((c >> 1) & 1));   // C has read stage c & 1 and Dt; the chain has read U
      if (tid == kStageLoader && c + 2 < nchunks && live()) tma_qk(c + 2);
      wait(B_P, par);
      if (tid == kOutIssuer && live()) {
        tc::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_PD, dadv(dP, ks * 32), dadv(dDl, ks * 2048), IDESC_PD, ks != 0);
        tc::mma_commit(bar(B_PD));
      }
      if (c + 1 < nchunks && warp == kOutIssuer / 32) {
        wait(B_TV, par ^ 1u);
        if (tid == kOutIssuer && live()) issue_u();
      }
      // ---- o = scale (Gam Y + P Delta), rows r < L ----
      wait(B_XY0 + s, (uint32_t)((c >> 1) & 1));
      wait(B_PD, par);
      tc::tc_fence_after();
      {
        float yv[32];
        const uint32_t ty = TM_XY + (uint32_t)s * 64;
        const float e2 = egam_r * y_scale;
#pragma unroll
        for (int k = 0; k < 2; ++k) {   // columns [32 half + 16 k, +16): Y and the four P Delta parts
          float y16[16], a0[16], a1[16], b0[16], b1[16];
          tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0 + 16, ty + 16 * k), y16);
          tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_PD + 16 * k), a0);
          tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_PD + 64 + 16 * k), a1);
          tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0 + 16, TM_PD + 16 * k), b0);
          tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0 + 16, TM_PD + 64 + 16 * k), b1);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) yv[16 * k + j] = p.scale * fmaf(e2, y16[j], (a0[j] + a1[j]) + (b0[j] + b1[j]));
        }
        if (L == 64) {   // row row64, columns [32 half, +32): one 128-byte row of half-tile `half`
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(sm + OFF_PO + (uint32_t)half * 8 * KB + tc::sw128(row64, 16 * q)) =
                make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
          tc::fence_proxy_async_smem();
        } else if (row64 < L) {   // a sequence's last chunk: rows past its end belong to others
          float4* out = reinterpret_cast<float4*>(p.o + ((t0 + c * 64 + row64) * p.Hv + h) * (int64_t)p.dv +
                                                  slab * 64 + half * 32);
#pragma unroll
          for (int j = 0; j < 32; j += 4) out[j >> 2] = make_float4(yv[j], yv[j + 1], yv[j + 2], yv[j + 3]);
        }
      }
      tc::tc_fence_before();
      if (wg_any(1, !live())) break;
      if (tid == 0) tc::mbar_arrive(bar(B_OD0 + s));   // Y of chunk c has been read
      if (tid == kStageLoader) {
        if (L == 64) {   // the tile is complete: one store, read back before the region is reused
          tc::tma_store_3d(&tout, sbase + OFF_PO, slab * 64, h, (int)(t0 + c * 64));
          tc::tma_store_3d(&tout, sbase + OFF_PO + 8 * KB, slab * 64 + 32, h, (int)(t0 + c * 64));
          tc::bulk_commit();
          tc::bulk_wait_read();
        }
        if (c + 1 < nchunks && live()) tma_p(c + 1);   // needed after the chain's next Delta
      }
    }
  } else {
    // ================================ chain warpgroup ================================
    const int ctid = tid - 128;
    const int64_t sb = ((int64_t)n * p.Hv + h) * 128 * p.dv + slab * 64;   // S[c][j] at sb + c dv + j
    // the state row of this thread: S[lane128][0..63] in registers, for the whole sequence
    float S[64];
    if (p.h0) {
      const float4* src = reinterpret_cast<const float4*>(p.h0 + sb + (int64_t)lane128 * p.dv);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 f = src[j];
        S[4 * j] = f.x; S[4 * j + 1] = f.y; S[4 * j + 2] = f.z; S[4 * j + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {   // the hi | lo operand
      uint4 h16, l16;
      split8(S + 8 * q, h16, l16);
      const uint32_t off = tc::sw128(lane128, 16 * q);
      st16(sm, OFF_SHI + off, h16);
      st16(sm, OFF_SHI + 16 * KB + off, l16);
    }
    if (ctid == 0) s_scale_slot[0] = 1.f;
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    wg_sync(2);
    bool s_exact = false;   // S0 operand holds exact codes with scale s_scale
    float s_scale = 1.f;
    // The registers S hold the state divided by sT: the E4M3 codes after a QDQ (sT = their scale),
    // plain values otherwise (sT = 1); the scale is folded into the next step's multiplier.
    float sT = 1.f;
    float i8s[2] = {0.f, 0.f};   // INT8: this row's two block scales of the last QDQ'd state
    for (int64_t c = 0; c < nchunks; ++c) {
      const int s = (int)(c & 1);
      const int L = chunk_len(c);
      const uint32_t par = (uint32_t)(c & 1);
      const uint32_t stg = (uint32_t)s * kStage;
      wait(B_QK0 + s, (uint32_t)((c >> 1) & 1));
      const float* vg = vecs(c);
      const float dr = vg[128 + row64], el = vg[64 + 63];
      const float f = vg[192] * s_scale;   // X = W S0 holds codes x codes: W scale x S0 scale
      if (!p.w_qdq) wait(B_WLO, par);
      if (c >= 2) wait(B_OD0 + s, (uint32_t)(((c - 2) >> 1) & 1));   // Y of chunk c - 2 has been read
      // ---- [X; Y] = [W; Q] S0 ----
      const uint32_t txy = TM_XY + (uint32_t)s * 64;
      if (ctid == kChainIssuer && live()) {
        tc::tc_fence_after();
        // [W codes or W hi; Q] x (S codes or S hi) [+ [W; Q] x S lo] [+ W lo x S hi]
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::mma_bf16(tmem + txy, dadv(dStgA, stg + (ks >> 2) * 16 * KB + (ks & 3) * 32), dadv(dS, ks * 2048),
                       IDESC_XY, ks > 0);
        if (!s_exact) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + txy, dadv(dStgA, stg + (ks >> 2) * 16 * KB + (ks & 3) * 32),
                         dadv(dS, 16 * KB + ks * 2048), IDESC_XY, 1);
        }
        if (!p.w_qdq) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_bf16(tmem + txy, dadv(dWlo, (ks >> 2) * 8 * KB + (ks & 3) * 32), dadv(dS, ks * 2048), IDESC_WLO, 1);
        }
        tc::mma_commit(bar(B_XY0 + s));
      }
      wait(B_XY0 + s, (uint32_t)((c >> 1) & 1));
      if (ctid == 96 && !p.w_qdq && c + 1 < nchunks && live()) tma_wlo(c + 1);   // W lo has been read
      // ---- Delta = U - f X, Dt = exp(gam_63 - gam_r) Delta ----
      wait(B_U, par);
      if (c > 0) wait(B_PD, (uint32_t)((c - 1) & 1));   // the previous P Delta has read Delta
      tc::tc_fence_after();
      float d[32];
      {
        float xv[32], uv[32], ulo[32];   // U = T''_hi V (lanes 0-15) + T''_lo V (lanes 16-31)
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, txy), xv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, txy + 16), xv + 16);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_U), uv);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_U + 16), uv + 16);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0 + 16, TM_U), ulo);
        tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0 + 16, TM_U + 16), ulo + 16);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) uv[j] += ulo[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float dt[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            d[8 * q + u] = fmaf(-f, xv[8 * q + u], uv[8 * q + u]);
            dt[u] = dr * d[8 * q + u];
          }
          uint4 h16, l16;
          split8(dt, h16, l16);
          const uint32_t off = tc::sw128(row64, 2 * (half * 32 + 8 * q));
          st16(sm, OFF_DL + 16 * KB + off, h16);
          st16(sm, OFF_DL + 24 * KB + off, l16);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      if (wg_any(2, !live())) break;
      if (ctid == kChainIssuer) {
        tc::tc_fence_after();
        // C = K^T [Dt hi | Dt lo] (N = 128: the two parts side by side)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_C, dadv(dStgM, stg + ks * 2048), dadv(dDl, 16 * KB + ks * 2048), IDESC_C, ks != 0);
        tc::mma_commit(bar(B_C));
      }
      // Delta hi | lo for the output warpgroup's P Delta (while C runs)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 h16, l16;
        split8(d + 8 * q, h16, l16);
        const uint32_t off = tc::sw128(row64, 2 * (half * 32 + 8 * q));
        st16(sm, OFF_DL + off, h16);
        st16(sm, OFF_DL + 8 * KB + off, l16);
      }
      tc::fence_proxy_async_smem();
      if (wg_any(2, !live())) break;
      if (ctid == 0) tc::mbar_arrive(bar(B_DRDY));
      // ---- S1 = Gam_63 S0 + C; QDQ at the 64-token boundary (Y read S0 with X, waited above) ----
      wait(B_C, par);
      if (ctid == 0) tc::mbar_arrive(bar(B_SF0 + s));   // [X; Y] and C have read stage s, U has been read
      tc::tc_fence_after();
      {
        float* const s1 = S;
        {
          const float elt = el * sT;
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // C = K^T Dt_hi + K^T Dt_lo, 16 columns at a time
            float ch[16], cl[16];
            tc::tmem_ld16(tc::tmem_addr(tmem, lane0, TM_C + 16 * k), ch);
            tc::tmem_ld16(tc::tmem_addr(tmem, lane0, TM_C + 64 + 16 * k), cl);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) s1[16 * k + j] = fmaf(elt, s1[16 * k + j], ch[j] + cl[j]);
          }
          sT = 1.f;
        }
        if (p.state_qdq == 1 && L == 64) {
          float m8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = fabsf(s1[u]);
#pragma unroll
          for (int j = 8; j < 64; ++j) m8[j & 7] = fmaxf(m8[j & 7], fabsf(s1[j]));
          float mm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          mm = warp_absmax(mm);
          if (lt == 0) red[quad] = mm;
          wg_sync(2);
          const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
          const float sS = qdq_scale(amax), rS = __frcp_rn(sS);
#pragma unroll
          for (int q = 0; q < 8; ++q) {   // the codes stay in S (dequantized as codes x sS)
#pragma unroll
            for (int u = 0; u < 8; u += 2) e4m3_codes2(s1[8 * q + u], s1[8 * q + u + 1], rS, s1[8 * q + u], s1[8 * q + u + 1]);
            st16(sm, OFF_SHI + tc::sw128(lane128, 16 * q), pack8(s1 + 8 * q));
          }
          s_exact = true;
          s_scale = sS;
          sT = sS;
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
            st16(sm, OFF_SHI + off, h16);
            st16(sm, OFF_SHI + 16 * KB + off, l16);
          }
          s_exact = false;
          s_scale = 1.f;
        }
      }
      if (ctid == 0) s_scale_slot[(c + 1) & 3] = s_scale;
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      if (wg_any(2, !live())) break;
    }
    if (live() && p.hT) {   // code x scale: the value the QDQ produced
      float4* out = reinterpret_cast<float4*>(p.hT + sb + (int64_t)lane128 * p.dv);
#pragma unroll
      for (int j = 0; j < 64; j += 4)
        out[j >> 2] = make_float4(__fmul_rn(S[j], sT), __fmul_rn(S[j + 1], sT), __fmul_rn(S[j + 2], sT),
                                  __fmul_rn(S[j + 3], sT));
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
      // TMA loads may still be landing in this CTA's shared memory: wait for each barrier's
      // current phase (one of the two parities returns at once), bounded
      const int tx_bars[5] = {B_QK0, B_QK1, B_TV, B_P, B_WLO};
      for (int i = 0; i < 5; ++i) {
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

bool chunk_split_supported(const ChunkProblem& p) { return p.dk == 128 && !p.kda && p.dv % 64 == 0; }

SplitLayout chunk_split_layout(const ChunkProblem& p) {
  SplitLayout l{};
  const int64_t tokens = (int64_t)p.B * p.T;
  l.slots = tokens / 64 + p.N;
  l.items = l.slots * p.Hv;
  l.wt_item_bytes = p.w_qdq ? 16 * KB : 32 * KB;
  auto up = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
  l.off_wt = up(kStatusBytes);
  l.off_tt = up(l.off_wt + (size_t)l.items * l.wt_item_bytes);
  l.off_p = up(l.off_tt + (size_t)l.items * 16 * KB);
  l.off_vec = up(l.off_p + (size_t)l.items * 16 * KB);
  l.off_order = up(l.off_vec + (size_t)l.items * 1024);
  l.total = l.off_order + (size_t)p.N * 4;
  return l;
}

const int32_t* stage_chain_order(const ChunkProblem& p, unsigned char* ws, size_t off_order, cudaStream_t stream,
                                 cudaError_t* err) {
  *err = cudaSuccess;
  if (p.N < 2 || !(p.lens ? p.lens_host != nullptr : (p.cu && p.cu_host))) return nullptr;
  std::vector<int32_t> order(p.N), len(p.N);
  for (int n = 0; n < p.N; ++n) {
    order[n] = n;
    len[n] = p.lens ? p.lens_host[n] : p.cu_host[n + 1] - p.cu_host[n];
  }
  const int32_t* l = len.data();
  std::stable_sort(order.begin(), order.end(), [l](int32_t a, int32_t b) { return l[a] > l[b]; });
  // pageable source: the copy is staged before the call returns, so the vector may go
  *err = cudaMemcpyAsync(ws + off_order, order.data(), (size_t)p.N * 4, cudaMemcpyHostToDevice, stream);
  return *err == cudaSuccess ? reinterpret_cast<const int32_t*>(ws + off_order) : nullptr;
}

cudaError_t launch_chunk_split(const ChunkProblem& p, void* ws, cudaStream_t stream) {
  const SplitLayout lay = chunk_split_layout(p);
  if (lay.items * 256 >= (int64_t)1 << 31) return cudaErrorInvalidValue;   // TMA row coordinates are int32
  unsigned char* w = static_cast<unsigned char*>(ws);
  cudaError_t e;
  // the chain order is staged first, so that the chain kernel directly follows the prep kernel
  const int32_t* order = stage_chain_order(p, w, lay.off_order, stream, &e);
  if (e != cudaSuccess) return e;
  e = launch_chunk_prep(p, lay, w, stream);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.N * p.Hv * (p.dv / 64);
  if (blocks == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  const int64_t tmap = tokens > 0 ? tokens : 1;   // an empty batch still needs valid maps (never loaded)
  CUtensorMap tq16, tk, tv, tw16, tw64, ttt, tpp, tout;
  const int64_t wrows = lay.items * (p.w_qdq ? 128 : 256);
  if (!make_bf16_map(&tq16, p.q, 128, p.Hqk, tmap, 16) || !make_bf16_map(&tk, p.k, 128, p.Hqk, tmap) ||
      !make_bf16_map(&tv, p.v, p.dv, p.Hv, tmap) || !make_bf16_rows_map(&tw16, w + lay.off_wt, wrows, 16) ||
      !make_bf16_rows_map(&tw64, w + lay.off_wt, wrows, 64) ||
      !make_bf16_rows_map(&ttt, w + lay.off_tt, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tpp, w + lay.off_p, lay.items * 128, 128) ||
      !make_f32_out_map(&tout, p.o, p.dv, p.Hv, tmap))
    return cudaErrorInvalidValue;
  ChainParams cp{order, reinterpret_cast<const float*>(w + lay.off_vec), p.h0, p.cu, p.lens, p.o, p.hT, reinterpret_cast<int*>(ws),
                 p.T, p.Hqk, p.Hv, p.dv, p.scale, p.state_qdq, p.w_qdq};
  cp.sscale = p.state_scales;
  e = cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the chain's CTAs may become resident while the prep's last
  // wave runs (griddepcontrol.wait in the kernel holds back every read of the staging)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chunk_chain_kernel, tq16, tk, tv, tw16, tw64, ttt, tpp, tout, cp);
}

}  // namespace gdn
