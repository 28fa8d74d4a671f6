// chunk_simt.cu -- chunked gated-delta-rule forward in fp32 on CUDA cores.
//
// One CTA per (sequence n, value head h, 64-column value slab); the CTA walks the
// sequence's 64-token chunks in order, carrying its [dk x 64] slice of S in shared memory.
// The slab is exactly one state-QDQ tile (all dk rows x 64 value columns, "GDN state/W QAT
// foundation", "What does this PR do?"), so the tile amax is CTA-local.
//
// Per chunk of L <= 64 tokens (rows r >= L are zero-padded: k = q = v = 0, beta = g = 0, so
// they contribute nothing and T is the identity there), with gam = prefix sums of g:
//   A[r][i]  = beta_r exp(gam_r - gam_i) (k_r . k_i),  i < r     (KDA: sum_c with per-channel gam)
//   P[r][i]  = exp(gam_r - gam_i) (q_r . k_i),        i <= r
//   T        = (I + A)^{-1}            16 x 16 diagonal blocks by forward substitution, then
//                                       T[b][c] = -T[b][b] sum_m A[b][m] T[m][c] by block rows
//   W        = T (beta exp(gam) K),  U = T (beta V);   W <- QDQ(W) over the chunk (W QDQ)
//   Delta    = U - W S0
//   o        = scale [ exp(gam) (Q S0) + P Delta ]
//   S1       = exp(gam_L) S0 + (K exp(gam_L - gam))^T Delta;  QDQ(S1) when L == 64 (state QDQ)
// Decays are always exponentials of non-positive prefix differences (the causal mask is
// applied before the exp), never a ratio of exponentials ("Add KDA prefill numerical
// emulation for QAT", "What does this PR do?").
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;
constexpr int SL = kStateTileCols;   // value columns per CTA

template <int DK, bool KDA>
struct SimtSmem {
  __nv_bfloat16 K[C][DK + 2];   // +2: odd word stride for transposed reads
  __nv_bfloat16 Q[C][DK + 2];
  float V[C][SL];
  float S[DK][SL];
  float Am[C][C + 1];
  float Tm[C][C + 1];
  float Pm[C][C + 1];
  float W[C][DK + 1];           // W, solve scratch, then decay-scaled K
  float D[C][SL];               // Delta
  float gam[KDA ? C * DK : C];  // prefix sums of g in the chunk
  float egam[C];                // GDN: exp(gam_r)
  float beta[C];
  float red[kThreads / 32];
};

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

template <int DK, bool KDA>
__global__ void __launch_bounds__(kThreads, 1) chunk_simt_kernel(ChunkProblem p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<SimtSmem<DK, KDA>*>(smem_raw);
  const int nslab = p.dv / SL;
  const int slab = blockIdx.x % nslab;
  const int h = (blockIdx.x / nslab) % p.Hv;
  const int n = blockIdx.x / (nslab * p.Hv);
  const int hq = h / (p.Hv / p.Hqk);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  int64_t t0, len;
  if (p.cu) {
    t0 = p.cu[n];
    len = (int64_t)p.cu[n + 1] - t0;
  } else {
    t0 = (int64_t)n * p.T;
    len = p.T;
  }
  if (p.lens) len = p.lens[n];
  const __nv_bfloat16* qg = (const __nv_bfloat16*)p.q;
  const __nv_bfloat16* kg = (const __nv_bfloat16*)p.k;
  const __nv_bfloat16* vg = (const __nv_bfloat16*)p.v;
  const int64_t sbase = ((int64_t)n * p.Hv + h) * DK * p.dv + slab * SL;

  for (int e = tid; e < DK * SL; e += kThreads) {
    const int c = e / SL, j = e % SL;
    sm.S[c][j] = p.h0 ? p.h0[sbase + (int64_t)c * p.dv + j] : 0.f;
  }

  constexpr int kTM = DK / 16;
  float last_s = 0.f, last_i8[kTM][2];   // scales of the last QDQ'd state (E4M3 tile; INT8 blocks)
#pragma unroll
  for (int a = 0; a < kTM; ++a) last_i8[a][0] = last_i8[a][1] = 0.f;
  for (int64_t c0 = 0; c0 < len; c0 += C) {
    const int L = (len - c0) < C ? (int)(len - c0) : C;
    __syncthreads();
    // ---- load the chunk (zero-padded past L) ----
    for (int e = tid; e < C * (DK / 8); e += kThreads) {
      const int r = e / (DK / 8), c8 = (e % (DK / 8)) * 8;
      uint4 kv = make_uint4(0, 0, 0, 0), qv = make_uint4(0, 0, 0, 0);
      if (r < L) {
        const int64_t off = ((t0 + c0 + r) * p.Hqk + hq) * DK + c8;
        kv = *reinterpret_cast<const uint4*>(kg + off);
        qv = *reinterpret_cast<const uint4*>(qg + off);
      }
      uint32_t* kd = reinterpret_cast<uint32_t*>(&sm.K[r][c8]);
      uint32_t* qd = reinterpret_cast<uint32_t*>(&sm.Q[r][c8]);
      kd[0] = kv.x; kd[1] = kv.y; kd[2] = kv.z; kd[3] = kv.w;
      qd[0] = qv.x; qd[1] = qv.y; qd[2] = qv.z; qd[3] = qv.w;
    }
    for (int e = tid; e < C * (SL / 8); e += kThreads) {
      const int r = e / (SL / 8), j8 = (e % (SL / 8)) * 8;
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (r < L) load_bf16x8(vg + ((t0 + c0 + r) * p.Hv + h) * p.dv + slab * SL + j8, f);
#pragma unroll
      for (int u = 0; u < 8; ++u) sm.V[r][j8 + u] = f[u];
    }
    if (tid < C) sm.beta[tid] = tid < L ? p.beta[(t0 + c0 + tid) * p.Hv + h] : 0.f;
    if (KDA) {
      if (tid < DK) {   // channel-wise prefix sums, in token order
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
          if (r < L) acc += p.g[((t0 + c0 + r) * p.Hv + h) * DK + tid];
          sm.gam[r * DK + tid] = acc;
        }
      }
    } else if (tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        if (r < L) acc += p.g[(t0 + c0 + r) * p.Hv + h];
        sm.gam[r] = acc;
      }
    }
    __syncthreads();
    if (!KDA && tid < C) sm.egam[tid] = expf(sm.gam[tid]);

    // ---- A and P (64 x 64, thread tile 4 x 4: r = ty + 16 a, i = tx + 16 b) ----
    {
      float accA[4][4] = {}, accP[4][4] = {};
      for (int c = 0; c < DK; ++c) {
        float kr[4], qr[4], ki[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          kr[a] = __bfloat162float(sm.K[ty + 16 * a][c]);
          qr[a] = __bfloat162float(sm.Q[ty + 16 * a][c]);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) ki[b] = __bfloat162float(sm.K[tx + 16 * b][c]);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int r = ty + 16 * a, i = tx + 16 * b;
            if (KDA) {
              if (i <= r) {
                const float e = __expf(sm.gam[r * DK + c] - sm.gam[i * DK + c]);
                accA[a][b] = fmaf(kr[a] * ki[b], e, accA[a][b]);
                accP[a][b] = fmaf(qr[a] * ki[b], e, accP[a][b]);
              }
            } else {
              accA[a][b] = fmaf(kr[a], ki[b], accA[a][b]);
              accP[a][b] = fmaf(qr[a], ki[b], accP[a][b]);
            }
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int r = ty + 16 * a, i = tx + 16 * b;
          float dec = 1.f;
          if (!KDA && i <= r) dec = __expf(sm.gam[r] - sm.gam[i]);
          sm.Am[r][i] = i < r ? sm.beta[r] * dec * accA[a][b] : 0.f;
          sm.Pm[r][i] = i <= r ? dec * accP[a][b] : 0.f;
        }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}: diagonal 16 x 16 blocks (one thread per block column) ----
    if (tid < C) {
      const int b0 = (tid >> 4) * 16, j = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) acc = fmaf(-sm.Am[b0 + r][b0 + i], x[i], acc);
        x[r] = r < j ? 0.f : acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sm.Tm[b0 + r][b0 + j] = x[r];
#pragma unroll
      for (int r = 0; r < 16; ++r)   // upper off-diagonal blocks of this block column are zero
        for (int bb = 0; bb < 4; ++bb)
          if (bb * 16 < b0) sm.Tm[bb * 16 + r][b0 + j] = 0.f;
    }
    __syncthreads();
    // block rows bi = 1..3: Y_bj = sum_{m = bj}^{bi - 1} A[bi][m] T[m][bj], T[bi][bj] = -T[bi][bi] Y_bj
    for (int bi = 1; bi < 4; ++bi) {
      const int rr = tid >> 4, cc = tid & 15;
      for (int bj = 0; bj < bi; ++bj) {
        float acc = 0.f;
        for (int m = bj * 16; m < bi * 16; ++m) acc = fmaf(sm.Am[bi * 16 + rr][m], sm.Tm[m][bj * 16 + cc], acc);
        sm.W[rr][bj * 16 + cc] = acc;
      }
      __syncthreads();
      for (int bj = 0; bj < bi; ++bj) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(sm.Tm[bi * 16 + rr][bi * 16 + m], sm.W[m][bj * 16 + cc], acc);
        sm.Tm[bi * 16 + rr][bj * 16 + cc] = -acc;
      }
      __syncthreads();
    }

    // ---- U = T (beta V) in registers (tile 4 x 4 over [64 x 64]) ----
    float acc[4][4] = {};
    for (int i = 0; i < C; ++i) {
      float ta[4], vb[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) ta[a] = sm.Tm[ty + 16 * a][i];
      const float bi = sm.beta[i];
#pragma unroll
      for (int b = 0; b < 4; ++b) vb[b] = bi * sm.V[i][tx + 16 * b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(ta[a], vb[b], acc[a][b]);
    }
    // ---- W = T (beta exp(gam) K) (tile 4 x DK/16 over [64 x DK]) ----
    {
      constexpr int TN = DK / 16;
      float wacc[4][TN] = {};
      for (int i = 0; i < C; ++i) {
        float ta[4], xb[TN];
#pragma unroll
        for (int a = 0; a < 4; ++a) ta[a] = sm.Tm[ty + 16 * a][i];
#pragma unroll
        for (int b = 0; b < TN; ++b) {
          const int c = tx + 16 * b;
          const float kd = __bfloat162float(sm.K[i][c]);
          xb[b] = KDA ? sm.beta[i] * __expf(sm.gam[i * DK + c]) * kd : sm.beta[i] * sm.egam[i] * kd;
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < TN; ++b) wacc[a][b] = fmaf(ta[a], xb[b], wacc[a][b]);
      }
      float wmax = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < TN; ++b) wmax = fmaxf(wmax, fabsf(wacc[a][b]));
      if (p.w_qdq) {   // one scale over the chunk's W (padded rows are zero)
        const float s = qdq_scale(block_max(wmax, sm.red));
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < TN; ++b) wacc[a][b] = qdq1(wacc[a][b], s);
      }
      __syncthreads();   // all reads of the solve scratch in W are done
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < TN; ++b) sm.W[ty + 16 * a][tx + 16 * b] = wacc[a][b];
    }
    __syncthreads();
    // ---- Delta = U - W S0 ----
    for (int c = 0; c < DK; ++c) {
      float wa[4], sb[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) wa[a] = sm.W[ty + 16 * a][c];
#pragma unroll
      for (int b = 0; b < 4; ++b) sb[b] = sm.S[c][tx + 16 * b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(-wa[a], sb[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) sm.D[ty + 16 * a][tx + 16 * b] = acc[a][b];
    __syncthreads();
    // ---- o = scale [exp(gam) (Q S0) + P Delta] ----
    {
      float oacc[4][4] = {};
      for (int c = 0; c < DK; ++c) {
        float qa[4], sb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int r = ty + 16 * a;
          qa[a] = __bfloat162float(sm.Q[r][c]);
          if (KDA) qa[a] *= __expf(sm.gam[r * DK + c]);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) sb[b] = sm.S[c][tx + 16 * b];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) oacc[a][b] = fmaf(qa[a], sb[b], oacc[a][b]);
      }
      if (!KDA) {
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) oacc[a][b] *= sm.egam[ty + 16 * a];
      }
      for (int i = 0; i < C; ++i) {
        float pa[4], db[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) pa[a] = sm.Pm[ty + 16 * a][i];
#pragma unroll
        for (int b = 0; b < 4; ++b) db[b] = sm.D[i][tx + 16 * b];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) oacc[a][b] = fmaf(pa[a], db[b], oacc[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = ty + 16 * a;
        if (r < L) {
          float* orow = p.o + ((t0 + c0 + r) * p.Hv + h) * (int64_t)p.dv + slab * SL;
#pragma unroll
          for (int b = 0; b < 4; ++b) orow[tx + 16 * b] = p.scale * oacc[a][b];
        }
      }
    }
    __syncthreads();   // all reads of W and S for this chunk are done
    // ---- decay-scaled keys Kd[i][c] = k_i[c] exp(gam_L[c] - gam_i[c]) into W ----
    for (int e = tid; e < C * DK; e += kThreads) {
      const int i = e / DK, c = e % DK;
      const float gl = KDA ? sm.gam[(C - 1) * DK + c] : sm.gam[C - 1];
      const float gi = KDA ? sm.gam[i * DK + c] : sm.gam[i];
      sm.W[i][c] = __bfloat162float(sm.K[i][c]) * __expf(gl - gi);
    }
    __syncthreads();
    // ---- S1 = exp(gam_L) S0 + Kd^T Delta (tile DK/16 x 4 over [DK x 64]) ----
    {
      constexpr int TM = DK / 16;
      float sacc[TM][4];
#pragma unroll
      for (int a = 0; a < TM; ++a) {
        const int c = ty + 16 * a;
        const float el = __expf(KDA ? sm.gam[(C - 1) * DK + c] : sm.gam[C - 1]);
#pragma unroll
        for (int b = 0; b < 4; ++b) sacc[a][b] = el * sm.S[c][tx + 16 * b];
      }
      for (int i = 0; i < C; ++i) {
        float ka[TM], db[4];
#pragma unroll
        for (int a = 0; a < TM; ++a) ka[a] = sm.W[i][ty + 16 * a];
#pragma unroll
        for (int b = 0; b < 4; ++b) db[b] = sm.D[i][tx + 16 * b];
#pragma unroll
        for (int a = 0; a < TM; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) sacc[a][b] = fmaf(ka[a], db[b], sacc[a][b]);
      }
      if (p.state_qdq == 1 && L == C) {   // the chunk ended on a 64-token boundary
        float m = 0.f;
#pragma unroll
        for (int a = 0; a < TM; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) m = fmaxf(m, fabsf(sacc[a][b]));
        const float s = qdq_scale(block_max(m, sm.red));
        last_s = s;
#pragma unroll
        for (int a = 0; a < TM; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) sacc[a][b] = qdq1(sacc[a][b], s);
      } else if (p.state_qdq == 2 && L == C) {
        // INT8 blocks of one key row x 32 value columns: row ty + 16 a, columns tx + 16 b, so
        // block 0 holds b = 0, 1 and block 1 b = 2, 3; the 16 threads of a row are the 16
        // consecutive lanes tx = 0..15 of one half-warp
#pragma unroll
        for (int a = 0; a < TM; ++a)
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            float m = fmaxf(fabsf(sacc[a][2 * blk]), fabsf(sacc[a][2 * blk + 1]));
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float sc = int8_scale(m), rc = __frcp_rn(sc);
            last_i8[a][blk] = sc;
            sacc[a][2 * blk] = int8_qdq_rcp(sacc[a][2 * blk], rc, sc);
            sacc[a][2 * blk + 1] = int8_qdq_rcp(sacc[a][2 * blk + 1], rc, sc);
          }
      }
#pragma unroll
      for (int a = 0; a < TM; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) sm.S[ty + 16 * a][tx + 16 * b] = sacc[a][b];
    }
  }
  __syncthreads();
  if (p.hT) {
    for (int e = tid; e < DK * SL; e += kThreads) {
      const int c = e / SL, j = e % SL;
      p.hT[sbase + (int64_t)c * p.dv + j] = sm.S[c][j];
    }
  }
  if (p.state_scales) {   // the final state was QDQ'd iff its last token was a 64th token
    const bool q = len > 0 && len % C == 0;
    const int64_t unit = (int64_t)n * p.Hv + h;
    if (p.state_qdq == 2) {
      if (tx == 0) {
#pragma unroll
        for (int a = 0; a < kTM; ++a) {
          float* dst = p.state_scales + (unit * DK + ty + 16 * a) * (p.dv / kInt8BlockCols) + slab * 2;
          dst[0] = q ? last_i8[a][0] : 0.f;
          dst[1] = q ? last_i8[a][1] : 0.f;
        }
      }
    } else if (tid == 0) {
      p.state_scales[unit * nslab + slab] = q ? last_s : 0.f;
    }
  }
}

template <int DK, bool KDA>
cudaError_t launch_t(const ChunkProblem& p, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<DK, KDA>);
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<DK, KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.N * p.Hv * (p.dv / SL);
  if (blocks == 0) return cudaSuccess;
  chunk_simt_kernel<DK, KDA><<<(unsigned)blocks, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkProblem& p, cudaStream_t stream) {
  if (p.dk == 64) return p.kda ? launch_t<64, true>(p, stream) : launch_t<64, false>(p, stream);
  if (p.dk == 128) return p.kda ? launch_t<128, true>(p, stream) : launch_t<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
