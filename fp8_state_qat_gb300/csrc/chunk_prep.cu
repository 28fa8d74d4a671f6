// chunk_prep.cu -- the state-independent half of the chunked gated-delta-rule forward (dk = 128),
// one CTA per (chunk, v-head) work item, all items in parallel.
//
// For chunk c of sequence n and v-head h (L <= 64 tokens; rows r >= L carry beta = g = 0 and so
// drop out), with gam = prefix sums of g inside the chunk and Gam = exp(gam):
//   G      [K; Q] K^T                              tcgen05 bf16, M=128 N=64 K=128 (exact products)
//   A      A[r][i] = beta_r exp(gam_r - gam_i) (k_r . k_i), i < r          (rows 0-63 of G)
//   P      P[r][i] = exp(gam_r - gam_i) (q_r . k_i), i <= r < L -> workspace as bf16 hi + lo rows,
//          interleaved (rows 64-127 of G)
//          The decays exp(gam_r - gam_i) are exp(gam_r - m) exp(m - gam_i) with m the midpoint of the
//          chunk's gam range while that range is at most 64 (both factors within e^+-32; 128
//          exponentials instead of 64 x 64), pairwise otherwise.
//   T      (I + A)^{-1} by blocked forward substitution: the two 32 x 32 diagonal blocks column by
//          column in registers (one thread per column, no barriers), then the block below the
//          diagonal, T10 = -T11 (A10 T00), as two 32 x 32 x 32 products over all threads
//   T''    T diag(beta)                 -> workspace as bf16 hi + lo rows, interleaved (the chain
//          forms U = T'' V)
//   W      T' K,  T' = T diag(beta Gam)            bf16 (T' as hi + lo), M=64 N=128 K=64
//   W QDQ  one E4M3 scale over the chunk's W; codes -> workspace (exact in bf16)
//   vec    gam, Gam, exp(gam_63 - gam), the W scale -> workspace
// ("GDN state/W QAT foundation", "What does this PR do?": W is the WY-transformed key block whose
// tile is quantized once per chunk; the decays are exponentials of non-positive prefix differences,
// "Add KDA prefill numerical emulation for QAT".) W is staged row-major per key block, so that the
// chain can stack its rows with Q's into one operand. The staged T'', P and W tiles are written
// to shared memory in the 128-byte swizzled layout and stored with TMA (plain row-major rows in the
// workspace; the chain's TMA loads apply the swizzle again).
//
// The solve stays on the CUDA cores: its products are 32 x 32 x 32, so a tensor-core form would add
// two TMEM round trips (MMA, load, bf16 hi/lo split, shared-memory store) to the item's latency
// for fewer fp32 instructions than those epilogues themselves issue.
//
// None of this depends on the state, so a chunk never waits for the one before it: the grid is
// (slots x v-heads) CTAs of 128 threads, four resident per SM. Every mbarrier wait is bounded;
// a CTA whose wait gives up records it in the status word, stores nothing more, waits (bounded)
// for its TMA load in flight, frees its TMEM and exits.
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
//   K0 | Q0 | K1 | Q1: bf16 [64 tok][64] each, key columns 0-63 (K0, Q0) | 64-127 (K1, Q1); rows
//   0-127 of one key block ([K; Q]) are the M = 128 operand of G. Once G is read the Q blocks hold
//   P hi (Q0) | lo (Q1) until their TMA store has read them, then T00 | T11 (Q0), T10 | scratch
//   (Q1) (fp32 [32][32] each), then T' hi (Q0) | lo (Q1). Once A is read its region holds T'' hi |
//   lo for its store; once the W MMA is done, K0 | K1 (| Q0 | Q1) hold the W rows for theirs.
constexpr uint32_t OFF_QK = 0;
constexpr uint32_t OFF_Q0 = 8 * KB, OFF_Q1 = 24 * KB;
constexpr uint32_t OFF_T00 = OFF_Q0, OFF_T11 = OFF_Q0 + 4 * KB, OFF_T10 = OFF_Q1, OFF_Y = OFF_Q1 + 4 * KB;
constexpr uint32_t OFF_A = 32 * KB;                    // A fp32 [64][68]
constexpr uint32_t OFF_VEC = OFF_A + 64 * A_LD * 4;    // gam, Gam, beta, e^(gam - m), e^(m - gam) [64]; 4 partial maxima; flag
constexpr uint32_t kSmemBytes = OFF_VEC + 5 * 256 + 64 + 1024;   // + slack to align the base
// four CTAs per SM: shared memory (with the 1 KB each CTA reserves) and TMEM columns fit
static_assert(4 * (kSmemBytes + 1024) <= 228 * KB, "four CTAs per SM no longer fit");

constexpr uint32_t TM_G = 0, TM_W = 0;   // W (128 columns) over G once G is read
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t IDESC_G = tc::make_idesc(tc::kKindBF16, 128, 64, false, false);
constexpr uint32_t IDESC_W = tc::make_idesc(tc::kKindBF16, 64, 128, false, true);

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

// Staged hi / lo pairs of 64-row matrices are interleaved in 16-row groups (rows 32 g .. 32 g + 15
// the hi rows 16 g .., rows 32 g + 16 .. the lo rows), so that the chain's one M = 128 product
// over both leaves hi . B in TMEM lanes 0-15 and lo . B in lanes 16-31 of each quadrant: the
// position of hi row r (lo row r: + 16).
__device__ __forceinline__ int ilv_row(int r) { return 32 * (r >> 4) + (r & 15); }

__device__ __forceinline__ int64_t seq_start(const PrepParams& p, int n) {
  return p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
}

__global__ void __launch_bounds__(kThreads, 4)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap twt, const __grid_constant__ CUtensorMap ttt,
                  const __grid_constant__ CUtensorMap tpp, const PrepParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[3];
  __shared__ uint32_t tmem_slot;

  // the state chain that follows may start its set-up (it waits for this grid before reading any
  // of its output)
  asm volatile("griddepcontrol.launch_dependents;");
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
  float* const T00 = reinterpret_cast<float*>(sm + OFF_T00);
  float* const T11 = reinterpret_cast<float*>(sm + OFF_T11);
  float* const T10 = reinterpret_cast<float*>(sm + OFF_T10);
  float* const Ym = reinterpret_cast<float*>(sm + OFF_Y);
  float* const vgam = reinterpret_cast<float*>(sm + OFF_VEC);
  float* const vegam = vgam + 64;
  float* const vbeta = vgam + 128;
  float* const vE = vgam + 192;      // exp(gam_r - m)
  float* const vF = vgam + 256;      // exp(m - gam_i)
  float* const red = vgam + 320;     // [4]
  int* const factored = reinterpret_cast<int*>(vgam + 324);
  const uint32_t bar_k = tc::smem_u32(&bars[0]), bar_g = tc::smem_u32(&bars[1]), bar_w = tc::smem_u32(&bars[2]);

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(tc::smem_u32(&bars[i]), 1);
    tc::mbar_fence_init();
    tc::mbar_expect_tx(bar_k, 32 * KB);
    tc::tma_load_3d(sbase + OFF_QK, &tk, bar_k, 0, hq, tok);
    tc::tma_load_3d(sbase + OFF_Q0, &tq, bar_k, 0, hq, tok);
    tc::tma_load_3d(sbase + OFF_QK + 16 * KB, &tk, bar_k, 64, hq, tok);
    tc::tma_load_3d(sbase + OFF_Q1, &tq, bar_k, 64, hq, tok);
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
    // the chunk's gam range (rows past L repeat the last prefix sum) and its midpoint anchor
    float mx = fmaxf(ga, gc), mn = fminf(ga, gc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    }
    const float m = 0.5f * (mx + mn);
    vE[lt] = __expf(ga - m); vE[lt + 32] = __expf(gc - m);
    vF[lt] = __expf(m - ga); vF[lt + 32] = __expf(m - gc);
    if (lt == 0) *factored = (mx - mn) <= 64.f;
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

  const uint64_t dQK = tc::make_sdesc(sbase + OFF_QK, 16, 1024);       // K-major [K; Q] / K rows
  const uint64_t dKn = tc::make_sdesc(sbase + OFF_QK, 16 * KB, 1024);  // MN-major K [i][c] (key blocks 16 KB apart)
  const uint64_t dTp = tc::make_sdesc(sbase + OFF_Q0, 16, 1024);       // K-major T' [r][i] (lo 16 KB on)

  bool ok = true;
  bool k_done = false;   // the Q / K tiles have landed (nothing left in flight on bar_k)
  float sW = 1.f;
  do {
    // ---- G = [K; Q] K^T ----
    if (warp == 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_k, 0));
    if (tid == 0 && ok) {
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 16 * KB + (ks & 3) * 32;
        tc::mma_bf16(tmem + TM_G, dadv(dQK, koff), dadv(dQK, koff), IDESC_G, ks > 0);
      }
      tc::mma_commit(bar_g);
    }
    if (__syncthreads_or(!ok)) break;
    k_done = true;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_g, 0));
    if (__syncthreads_or(!ok)) break;
    tc::tc_fence_after();

    // ---- A (threads 0-63: row r = tid of K K^T) and P (threads 64-127: row r = tid - 64 of Q K^T) ----
    {
      const int r = tid & 63;
      const bool is_a = tid < 64;
      // row factor and decays: A rows carry beta_r, P rows only their own rows r < L
      const float rowf = is_a ? vbeta[r] : (r < L ? 1.f : 0.f);
      const bool fac = *factored != 0;
      const float er = rowf * vE[r], gr = vgam[r];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {   // columns [32 hb, 32 hb + 32)
        float v[32];
        ld32(tmem, lane0, TM_G + 32 * hb, v);
        if (fac) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(vF + 32 * hb + i);
            v[i] *= er * f.x; v[i + 1] *= er * f.y; v[i + 2] *= er * f.z; v[i + 3] *= er * f.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)   // the exponent is clamped so both select inputs are finite
            v[i] *= rowf * __expf(fminf(gr - vgam[32 * hb + i], 0.f));
        }
        if (is_a) {   // strictly lower part, fp32
          float4* dst = reinterpret_cast<float4*>(Am + r * A_LD + 32 * hb);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const int c = 32 * hb + j;
            dst[j >> 2] = make_float4(c < r ? v[j] : 0.f, c + 1 < r ? v[j + 1] : 0.f, c + 2 < r ? v[j + 2] : 0.f,
                                      c + 3 < r ? v[j + 3] : 0.f);
          }
        } else {      // lower part with the diagonal, bf16 hi | lo rows interleaved (K-major [row][i])
          const int ah = ilv_row(r), al = ah + 16;
          const uint32_t rh = (ah < 64 ? OFF_Q0 : OFF_Q1), rl = (al < 64 ? OFF_Q0 : OFF_Q1);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float x8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x8[u] = 32 * hb + 8 * q + u <= r ? v[8 * q + u] : 0.f;
            uint4 h16, l16;
            split8(x8, h16, l16);
            st16(sm, rh + tc::sw128(ah & 63, 64 * hb + 16 * q), h16);
            st16(sm, rl + tc::sw128(al & 63, 64 * hb + 16 * q), l16);
          }
        }
      }
      if (!is_a) tc::fence_proxy_async_smem();
    }
    __syncthreads();   // A and the P tile complete; G (and with it the Q tiles) fully read
    if (tid == 64) {   // P hi | lo -> workspace rows item * 128 + [0, 64) | [64, 128)
      tc::tma_store_2d(&tpp, sbase + OFF_Q0, 0, (int)(item * 128));
      tc::tma_store_2d(&tpp, sbase + OFF_Q1, 0, (int)(item * 128 + 64));
      tc::bulk_commit();
    }

    // ---- T = (I + A)^{-1}, blocks of 32: T00, T11 one column per thread (warps 0, 1) ----
    if (warp < 2) {
      const int b0 = warp * 32, j = lt;
      float t[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float* arow = Am + (b0 + r) * A_LD + b0;
        float a0 = (r == j) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;   // split accumulators
#pragma unroll
        for (int i = 0; i < r; i += 4) {
          const float4 a = *reinterpret_cast<const float4*>(arow + i);
          a0 = fmaf(-a.x, t[i], a0);
          if (i + 1 < r) a1 = fmaf(-a.y, t[i + 1], a1);
          if (i + 2 < r) a2 = fmaf(-a.z, t[i + 2], a2);
          if (i + 3 < r) a3 = fmaf(-a.w, t[i + 3], a3);
        }
        t[r] = (a0 + a1) + (a2 + a3);
      }
      tc::named_bar_sync(1, 96);   // with warp 2: the P store has read the Q blocks
      float* Tb = warp == 0 ? T00 : T11;
#pragma unroll
      for (int r = 0; r < 32; ++r) Tb[r * 32 + j] = t[r];
    } else if (warp == 2) {
      if (tid == 64) tc::bulk_wait_read();
      tc::named_bar_sync(1, 96);
    }
    __syncthreads();
    {
      // thread (column j, rows 8 q .. 8 q + 7) of Y = A10 T00, then of T10 = -T11 Y
      const int j = lt, r0 = warp * 8;
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int i = 0; i < 32; i += 4) {
        const float t0 = T00[i * 32 + j], t1 = T00[(i + 1) * 32 + j], t2 = T00[(i + 2) * 32 + j],
                    t3 = T00[(i + 3) * 32 + j];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 a = *reinterpret_cast<const float4*>(Am + (32 + r0 + u) * A_LD + i);
          y[u] = fmaf(a.x, t0, fmaf(a.y, t1, fmaf(a.z, t2, fmaf(a.w, t3, y[u]))));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) Ym[(r0 + u) * 32 + j] = y[u];
      __syncthreads();
#pragma unroll
      for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 2
      for (int m = 0; m < 32; m += 4) {
        const float y0 = Ym[m * 32 + j], y1 = Ym[(m + 1) * 32 + j], y2 = Ym[(m + 2) * 32 + j], y3 = Ym[(m + 3) * 32 + j];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 t = *reinterpret_cast<const float4*>(T11 + (r0 + u) * 32 + m);
          y[u] = fmaf(t.x, y0, fmaf(t.y, y1, fmaf(t.z, y2, fmaf(t.w, y3, y[u]))));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) T10[(r0 + u) * 32 + j] = -y[u];
    }
    __syncthreads();

    // ---- T'' = T diag(beta) -> workspace, T' = T'' diag(Gam) -> the Q blocks (bf16 hi | lo,
    // [r][i]), which hold T: every thread reads its T entries before any writes ----
    // Two rounds of two row-quarters each, rows 32-63 first: T' hi row r lands on the bytes of T's
    // row r (T00 | T11 in Q0), T' lo rows 0-31 on T10 (T's rows 32-63, Q1), T' lo rows 32-63 on
    // the dead scratch, so each round reads its T rows, waits for every thread, then writes.
#pragma unroll
    for (int round = 0; round < 2; ++round) {
      float tv[2][8];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int task = tid + (t + 2 - 2 * round) * kThreads, r = task >> 3, i0 = (task & 7) * 8;
        const float* src = r < 32 ? (i0 < 32 ? T00 + r * 32 + i0 : nullptr)
                                  : (i0 < 32 ? T10 + (r - 32) * 32 + i0 : T11 + (r - 32) * 32 + (i0 - 32));
        if (src) {
          const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
          tv[t][0] = a.x; tv[t][1] = a.y; tv[t][2] = a.z; tv[t][3] = a.w;
          tv[t][4] = b.x; tv[t][5] = b.y; tv[t][6] = b.z; tv[t][7] = b.w;
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) tv[t][u] = 0.f;
        }
      }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int task = tid + (t + 2 - 2 * round) * kThreads, r = task >> 3, i0 = (task & 7) * 8;
        float t2[8], t1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          t2[u] = tv[t][u] * vbeta[i0 + u];
          t1[u] = t2[u] * vegam[i0 + u];
        }
        uint4 h16, l16;
        const uint32_t off = tc::sw128(r, 2 * i0);
        split8(t2, h16, l16);                  // T'' hi | lo rows interleaved in the A region (A is dead)
        st16(sm, OFF_A + tc::sw128(ilv_row(r), 2 * i0), h16);
        st16(sm, OFF_A + tc::sw128(ilv_row(r) + 16, 2 * i0), l16);
        split8(t1, h16, l16);
        st16(sm, OFF_Q0 + off, h16);
        st16(sm, OFF_Q1 + off, l16);
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 96) {   // not the MMA issuer: its MMAs would queue behind this copy
      tc::tma_store_2d(&ttt, sbase + OFF_A, 0, (int)(item * 128));   // T'' hi | lo
      tc::bulk_commit();
    }
    if (tid == 0) {
      tc::tc_fence_after();
      // W = T' K: A = T' hi / lo (K-major [r][i]), B = K (MN-major [i][c], key blocks 16 KB apart)
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_bf16(tmem + TM_W, dadv(dTp, part * 16 * KB + ks * 32), dadv(dKn, ks * 2048), IDESC_W, (part | ks) != 0);
      tc::mma_commit(bar_w);
    }
    ok = __all_sync(0xffffffffu, tc::mbar_wait(bar_w, 0));
    if (__syncthreads_or(!ok)) break;
    tc::tc_fence_after();

    // ---- W QDQ: thread = (row r = 16 warp + lane % 16, key block b = lane / 16), W[r][64 b .. 64 b + 63] ----
    {
      const int wr = warp * 16 + (lt & 15), wb = lt >> 4;
      float w[64];
#pragma unroll
      for (int k = 0; k < 4; ++k) tc::tmem_ld16x2<64>(tc::tmem_addr(tmem, lane0, TM_W + 16 * k), w + 16 * k);
      tc::tmem_ld_wait();
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
        // key block 0 -> K0, 1 -> K1 (both free once the W MMA is done)
        const uint32_t base = wb ? 16u * KB : 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float cd[8], dq[8];
#pragma unroll
          for (int u = 0; u < 8; u += 2) qdq_pair(w[8 * q + u], w[8 * q + u + 1], rW, sW, cd[u], cd[u + 1], dq[u], dq[u + 1]);
          st16(sm, base + tc::sw128(wr, 16 * q), pack8(cd));
        }
      } else {   // hi blocks -> K0 | K1, lo blocks -> Q0 | Q1
        const uint32_t base = wb ? 16u * KB : 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 h16, l16;
          split8(w + 8 * q, h16, l16);
          st16(sm, base + tc::sw128(wr, 16 * q), h16);
          st16(sm, base + 8 * KB + tc::sw128(wr, 16 * q), l16);
        }
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      if (p.w_qdq) {
        tc::tma_store_2d(&twt, sbase + 0, 0, (int)(item * 128));
        tc::tma_store_2d(&twt, sbase + 16 * KB, 0, (int)(item * 128 + 64));
      } else {
        tc::tma_store_2d(&twt, sbase + 0, 0, (int)(item * 256));
        tc::tma_store_2d(&twt, sbase + 16 * KB, 0, (int)(item * 256 + 64));
        tc::tma_store_2d(&twt, sbase + 8 * KB, 0, (int)(item * 256 + 128));
        tc::tma_store_2d(&twt, sbase + 24 * KB, 0, (int)(item * 256 + 192));
      }
      tc::bulk_commit();
      p.vec[item * 256 + 192] = sW;
    }
  } while (0);

  if (!ok) {
    if (tid == 0) {
      atomicExch(p.status, 1);
      if (!k_done) tc::mbar_wait(bar_k, 0, 1u << 16);   // the Q / K tiles may still be landing
    }
  }
  if (tid == 0 || tid == 64 || tid == 96) tc::bulk_wait_read();   // the stores have read their sources
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_prep(const ChunkProblem& p, const SplitLayout& lay, unsigned char* ws, cudaStream_t stream) {
  if (lay.items == 0) return cudaSuccess;
  const int64_t tokens = (int64_t)p.B * p.T;
  CUtensorMap tq, tk, twt, ttt, tpp;
  if (!make_bf16_map(&tq, p.q, 128, p.Hqk, tokens > 0 ? tokens : 1) ||
      !make_bf16_map(&tk, p.k, 128, p.Hqk, tokens > 0 ? tokens : 1) ||
      !make_bf16_rows_map(&twt, ws + lay.off_wt, lay.items * (p.w_qdq ? 128 : 256), 64) ||
      !make_bf16_rows_map(&ttt, ws + lay.off_tt, lay.items * 128, 128) ||
      !make_bf16_rows_map(&tpp, ws + lay.off_p, lay.items * 128, 64))
    return cudaErrorInvalidValue;
  PrepParams pp{p.g, p.beta, p.cu, p.lens, reinterpret_cast<float*>(ws + lay.off_vec), reinterpret_cast<int*>(ws),
                p.T, p.N, p.Hqk, p.Hv, p.w_qdq};
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  chunk_prep_kernel<<<(unsigned)lay.items, kThreads, kSmemBytes, stream>>>(tq, tk, twt, ttt, tpp, pp);
  return cudaGetLastError();
}

}  // namespace gdn
