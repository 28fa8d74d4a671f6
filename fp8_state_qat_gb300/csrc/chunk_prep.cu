// chunk_prep.cu -- the state-independent half of the chunked gated-delta-rule forward (dk = 128),
// one CTA per (chunk, v-head) work item, all items in parallel.
//
// For chunk c of sequence n and v-head h (L <= 64 tokens; rows r >= L carry beta = g = 0 and so
// drop out), with gam = prefix sums of g inside the chunk and Gam = exp(gam):
//   G      K K^T                                   tcgen05 bf16, M=64 N=64 K=128 (exact products)
//   A      A[r][i] = beta_r exp(gam_r - gam_i) (k_r . k_i), i < r
//   T      (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then three levels of
//          the off-diagonal block recurrence (CUDA cores, fp32)
//   T''    T diag(beta)                 -> workspace as bf16 hi + lo (the chain forms U = T'' V)
//   W^T    K^T T'^T,  T' = T diag(beta Gam)        bf16 (T' as hi + lo), M=128 N=64 K=64
//   W QDQ  one E4M3 scale over the chunk's W; codes -> workspace (exact in bf16)
//   vec    gam, Gam, exp(gam_63 - gam), the W scale -> workspace
// ("GDN state/W QAT foundation", "What does this PR do?": W is the WY-transformed key block whose
// tile is quantized once per chunk; the decays are exponentials of non-positive prefix differences,
// "Add KDA prefill numerical emulation for QAT".) W is produced transposed so that the QDQ epilogue
// uses all 128 TMEM lanes (one key channel per thread).
//
// None of this depends on the state, so a chunk never waits for the one before it: the grid is
// (slots x v-heads) CTAs of 128 threads, four resident per SM. Every mbarrier wait is bounded;
// a CTA whose wait gives up records it in the status word, stores nothing, waits (bounded) for its
// TMA load in flight, frees its TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t KB = 1024;
constexpr uint32_t A_LD = 68;
// shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_K = 0;                          // K tile: key columns 0-63 | 64-127, [64 tok][64] bf16 each
constexpr uint32_t OFF_A = 16 * KB;                    // A fp32 [64][68]; after the solve: T'' hi | lo
constexpr uint32_t OFF_T = 34 * KB;                    // T fp32 [64][68]
constexpr uint32_t OFF_SCR = OFF_T + 64 * A_LD * 4;    // solve scratch, 3 x 16 x 16 fp32
constexpr uint32_t OFF_W = OFF_T;                      // T' hi | lo over T once T is read; after the W MMA: W^T codes (or hi)
constexpr uint32_t OFF_VEC = OFF_SCR + 3 * KB;         // gam, Gam, beta [64]; 4 partial maxima
constexpr uint32_t kSmemBytes = OFF_VEC + 3 * 256 + 64 + 1024;   // + slack to align the base
static_assert(OFF_W + 16 * KB <= OFF_SCR, "T' overlaps the solve scratch");
// four CTAs per SM: shared memory (with the 1 KB each CTA reserves) and TMEM columns fit exactly
static_assert(4 * (kSmemBytes + 1024) <= 228 * KB, "four CTAs per SM no longer fit");

constexpr uint32_t TM_G = 0, TM_WT = 64;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t IDESC_G = tc::make_idesc(tc::kKindBF16, 64, 64, false, false);
constexpr uint32_t IDESC_WT = tc::make_idesc(tc::kKindBF16, 128, 64, true, false);

struct PrepParams {
  const float* g;
  const float* beta;
  const int32_t* cu;
  const int32_t* lens;   // tokens run per sequence, or null (whole sequences)
  float* vec;
  int* status;
  int T, N, Hqk, Hv;
  int w_qdq;
};

__device__ __forceinline__ int64_t seq_start(const PrepParams& p, int n) {
  return p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
}

__global__ void __launch_bounds__(kThreads, 4)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap twt,
                  const __grid_constant__ CUtensorMap ttt, const PrepParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[3];
  __shared__ uint32_t tmem_slot;

  const int64_t item = blockIdx.x;
  const int h = (int)(item % p.Hv);
  const int64_t slot = item / p.Hv;
  // the sequence owning this slot: the last n with floor(cu[n] / 64) + n <= slot
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_start(p, mid) / 64 + mid <= slot) lo = mid;
    else hi = mid - 1;
  }
  const int n = lo;
  const int64_t t0 = seq_start(p, n), len = p.lens ? (int64_t)p.lens[n] : seq_start(p, n + 1) - t0;
  const int64_t c = slot - (t0 / 64 + n);
  if (c < 0 || c * 64 >= len) return;   // no chunk uses this slot (uniform across the CTA)
  const int L = (int)(len - c * 64 < 64 ? len - c * 64 : 64);
  const int hq = h / (p.Hv / p.Hqk);
  const int tok = (int)(t0 + c * 64);

  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lt = tid & 31;
  const uint32_t lane0 = (uint32_t)warp * 32u;
  float* const Am = reinterpret_cast<float*>(sm + OFF_A);
  float* const Tm = reinterpret_cast<float*>(sm + OFF_T);
  float* const scr = reinterpret_cast<float*>(sm + OFF_SCR);
  float* const vgam = reinterpret_cast<float*>(sm + OFF_VEC);
  float* const vegam = vgam + 64;
  float* const vbeta = vgam + 128;
  float* const red = vgam + 192;
  const uint32_t bar_k = tc::smem_u32(&bars[0]), bar_g = tc::smem_u32(&bars[1]), bar_w = tc::smem_u32(&bars[2]);

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(tc::smem_u32(&bars[i]), 1);
    tc::mbar_fence_init();
    tc::mbar_expect_tx(bar_k, 16 * KB);
    tc::tma_load_3d(sbase + OFF_K, &tk, bar_k, 0, hq, tok);
    tc::tma_load_3d(sbase + OFF_K + 8 * KB, &tk, bar_k, 64, hq, tok);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
  if (warp == 1) {   // gates: prefix sums of g in the chunk, Gam, decay to the chunk end, beta
    const int64_t gb = (int64_t)tok * p.Hv + h;
    float ga = lt < L ? p.g[gb + (int64_t)lt * p.Hv] : 0.f;
    float gc = lt + 32 < L ? p.g[gb + (int64_t)(lt + 32) * p.Hv] : 0.f;
    const float ba = lt < L ? p.beta[gb + (int64_t)lt * p.Hv] : 0.f;
    const float bb = lt + 32 < L ? p.beta[gb + (int64_t)(lt + 32) * p.Hv] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ya = __shfl_up_sync(0xffffffffu, ga, off);
      const float yc = __shfl_up_sync(0xffffffffu, gc, off);
      if (lt >= off) { ga += ya; gc += yc; }
    }
    gc += __shfl_sync(0xffffffffu, ga, 31);
    const float gl = __shfl_sync(0xffffffffu, gc, 31);
    const float ea = __expf(ga), ec = __expf(gc), da = __expf(gl - ga), dc = __expf(gl - gc);
    vgam[lt] = ga; vgam[lt + 32] = gc;
    vegam[lt] = ea; vegam[lt + 32] = ec;
    vbeta[lt] = ba; vbeta[lt + 32] = bb;
    float* gv = p.vec + item * 256;
    gv[lt] = ga; gv[lt + 32] = gc;
    gv[64 + lt] = ea; gv[96 + lt] = ec;
    gv[128 + lt] = da; gv[160 + lt] = dc;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  const uint64_t dK = tc::make_sdesc(sbase + OFF_K, 16, 1024);         // K-major [tok][c]
  const uint64_t dKt = tc::make_sdesc(sbase + OFF_K, 8 * KB, 1024);    // MN-major K^T
  const uint64_t dTp = tc::make_sdesc(sbase + OFF_W, 16, 1024);        // K-major T' [r][i]

  bool ok = true;
  bool k_done = false;   // the K tile has landed (nothing left in flight on bar_k)
  float sW = 1.f;
  do {
    // ---- G = K K^T ----
    if (warp == 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_k, 0));
    if (tid == 0 && ok) {
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 8 * KB + (ks & 3) * 32;
        tc::mma_bf16(tmem + TM_G, dadv(dK, koff), dadv(dK, koff), IDESC_G, ks > 0);
      }
      tc::mma_commit(bar_g);
    }
    if (__syncthreads_or(!ok)) break;
    k_done = true;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_g, 0));
    if (__syncthreads_or(!ok)) break;
    tc::tc_fence_after();

    // ---- A (M = 64 accumulator: row 16 w + t % 16, columns 32 (t / 16) .. + 31) ----
    {
      const int r = warp * 16 + (lt & 15), half = lt >> 4;
      float v[32];
      tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_G), v);
      tc::tmem_ld16x2<32>(tc::tmem_addr(tmem, lane0, TM_G + 16), v + 16);
      tc::tmem_ld_wait();
      const float gr = vgam[r], br = vbeta[r];
      float4* dst = reinterpret_cast<float4*>(Am + r * A_LD + half * 32);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float a4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {   // the exponent is clamped so both select inputs are finite
          const int i = half * 32 + j + u;
          const float e = br * __expf(fminf(gr - vgam[i], 0.f)) * v[j + u];
          a4[u] = i < r ? e : 0.f;
        }
        dst[j >> 2] = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then the blocks
    // below the diagonal by levels of T_ij = -T_ii sum_{j <= m < i} A_im T_mj ----
    if (tid < 64) {
      const int b0 = (tid >> 4) * 16, jj = tid & 15;
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
#pragma unroll
      for (int r = 0; r < 16; ++r)
#pragma unroll
        for (int bb = 1; bb < 4; ++bb)
          if (bb * 16 > b0) Tm[(b0 + r) * A_LD + bb * 16 + jj] = 0.f;
    }
    __syncthreads();
    {
      // one 1 x 8 tile (row rr, columns c8 .. c8 + 7) of a 16 x 16 block per thread
      const int blk = tid >> 5, rr = (tid >> 1) & 15, c8 = (tid & 1) * 8;
      auto ytile = [&](int bi, int bj, float* y) {
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 4
        for (int m = 0; m < 16 * (bi - bj); ++m) {
          const float a = Am[(bi * 16 + rr) * A_LD + bj * 16 + m];
          const float4 ta = *reinterpret_cast<const float4*>(Tm + (bj * 16 + m) * A_LD + bj * 16 + c8);
          const float4 tb = *reinterpret_cast<const float4*>(Tm + (bj * 16 + m) * A_LD + bj * 16 + c8 + 4);
          y[0] = fmaf(a, ta.x, y[0]); y[1] = fmaf(a, ta.y, y[1]); y[2] = fmaf(a, ta.z, y[2]); y[3] = fmaf(a, ta.w, y[3]);
          y[4] = fmaf(a, tb.x, y[4]); y[5] = fmaf(a, tb.y, y[5]); y[6] = fmaf(a, tb.z, y[6]); y[7] = fmaf(a, tb.w, y[7]);
        }
      };
      auto put = [&](float* Y, const float* y) {
        *reinterpret_cast<float4*>(Y + rr * 16 + c8) = make_float4(y[0], y[1], y[2], y[3]);
        *reinterpret_cast<float4*>(Y + rr * 16 + c8 + 4) = make_float4(y[4], y[5], y[6], y[7]);
      };
      auto ttile = [&](int bi, int bj, const float* Y) {
        float t8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int m = 0; m < 16; ++m) {
          const float a = Tm[(bi * 16 + rr) * A_LD + bi * 16 + m];
          const float4 ya = *reinterpret_cast<const float4*>(Y + m * 16 + c8);
          const float4 yb = *reinterpret_cast<const float4*>(Y + m * 16 + c8 + 4);
          t8[0] = fmaf(a, ya.x, t8[0]); t8[1] = fmaf(a, ya.y, t8[1]); t8[2] = fmaf(a, ya.z, t8[2]); t8[3] = fmaf(a, ya.w, t8[3]);
          t8[4] = fmaf(a, yb.x, t8[4]); t8[5] = fmaf(a, yb.y, t8[5]); t8[6] = fmaf(a, yb.z, t8[6]); t8[7] = fmaf(a, yb.w, t8[7]);
        }
        float* dst = Tm + (bi * 16 + rr) * A_LD + bj * 16 + c8;
        *reinterpret_cast<float4*>(dst) = make_float4(-t8[0], -t8[1], -t8[2], -t8[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(-t8[4], -t8[5], -t8[6], -t8[7]);
      };
      float y[8];
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

    // ---- T'' = T diag(beta) -> the A region, T' = T'' diag(Gam) -> the W region (bf16 hi | lo, [r][i]),
    // which lies over T: every thread reads its T entries before any writes ----
    float4 tr[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int task = tid + t * kThreads, r = task >> 3, i0 = (task & 7) * 8;
      tr[2 * t] = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0);
      tr[2 * t + 1] = *reinterpret_cast<const float4*>(Tm + r * A_LD + i0 + 4);
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int task = tid + t * kThreads, r = task >> 3, i0 = (task & 7) * 8;
      const float4 ta = tr[2 * t], tb = tr[2 * t + 1];
      const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
      float t2[8], t1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        t2[u] = tv[u] * vbeta[i0 + u];
        t1[u] = t2[u] * vegam[i0 + u];
      }
      const uint32_t off = tc::sw128(r, 2 * i0);
      uint4 h16, l16;
      split8(t2, h16, l16);
      st16(sm, OFF_A + off, h16);
      st16(sm, OFF_A + 8 * KB + off, l16);
      split8(t1, h16, l16);
      st16(sm, OFF_W + off, h16);
      st16(sm, OFF_W + 8 * KB + off, l16);
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tma_store_2d(&ttt, sbase + OFF_A, 0, (int)(item * 128));   // T'' hi (rows 0-63) | lo (64-127)
      tc::bulk_commit();
      tc::tc_fence_after();
      // W^T = K^T T'^T: A = K^T (MN-major, key blocks 8 KB apart), B = T' hi / lo (K-major [r][i])
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_WT, dadv(dKt, ks * 2048), dadv(dTp, part * 8 * KB + ks * 32), IDESC_WT,
                       (part | ks) != 0);
      tc::mma_commit(bar_w);
    }
    ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_w, 0));
    if (__syncthreads_or(!ok)) break;
    tc::tc_fence_after();

    // ---- W QDQ: thread = key channel c (TMEM lane), its 64 values W[r][c] ----
    {
      float w[64];
      ld32(tmem, lane0, TM_WT, w);
      ld32(tmem, lane0, TM_WT + 32, w + 32);
      if (p.w_qdq) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) m = fmaxf(m, fabsf(w[j]));
        m = warp_max(m);
        if (lt == 0) red[warp] = m;
        __syncthreads();
        const float amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        sW = qdq_scale(amax);
        const float rW = __frcp_rn(sW);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float cd[8], dq[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2) qdq_pair(w[8 * q + u], w[8 * q + u + 1], rW, sW, cd[u], cd[u + 1], dq[u], dq[u + 1]);
          st16(sm, OFF_W + tc::sw128(tid, 16 * q), pack8(cd));
        }
      } else {   // hi -> the W region, lo -> the K region (both MMAs that read them are done)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 h16, l16;
          split8(w + 8 * q, h16, l16);
          st16(sm, OFF_W + tc::sw128(tid, 16 * q), h16);
          st16(sm, OFF_K + tc::sw128(tid, 16 * q), l16);
        }
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (p.w_qdq) {
        tc::tma_store_2d(&twt, sbase + OFF_W, 0, (int)(item * 128));
      } else {
        tc::tma_store_2d(&twt, sbase + OFF_W, 0, (int)(item * 256));
        tc::tma_store_2d(&twt, sbase + OFF_K, 0, (int)(item * 256 + 128));
      }
      tc::bulk_commit();
      p.vec[item * 256 + 192] = sW;
    }
  } while (0);

  if (!ok) {
    if (tid == 0) {
      atomicExch(p.status, 1);
      if (!k_done) tc::mbar_wait(bar_k, 0, 1u << 16);   // the K tile may still be landing
    }
  }
  if (tid == 0) tc::bulk_wait_read();   // the stores have read their shared-memory sources
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_prep(const ChunkProblem& p, const SplitLayout& lay, unsigned char* ws, cudaStream_t stream) {
  if (lay.items == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  CUtensorMap tk, twt, ttt;
  if (!make_bf16_map(&tk, p.k, 128, p.Hqk, tokens > 0 ? tokens : 1) ||
      !make_bf16_rows_map(&twt, ws + lay.off_wt, lay.items * (p.w_qdq ? 128 : 256), 128) ||
      !make_bf16_rows_map(&ttt, ws + lay.off_tt, lay.items * 128, 128))
    return cudaErrorInvalidValue;
  PrepParams pp{p.g, p.beta, p.cu, p.lens, reinterpret_cast<float*>(ws + lay.off_vec), reinterpret_cast<int*>(ws),
                p.T, p.N, p.Hqk, p.Hv, p.w_qdq};
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_prep_kernel<<<(unsigned)lay.items, kThreads, kSmemBytes, stream>>>(tk, twt, ttt, pp);
  return cudaGetLastError();
}

}  // namespace gdn
