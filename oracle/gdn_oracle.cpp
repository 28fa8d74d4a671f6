// gdn_oracle.cpp -- plain, slow, fp64 CPU oracle for the chunked gated-delta-rule
// forward with dynamic FP8 E4M3 fake quantize-dequantize (QDQ) of the recurrent state.
//
// TEST INFRASTRUCTURE ONLY. This file is the independent reference that the CUDA
// library is checked against. Only the tests, the smoke check and the CPU-baseline
// leg of the benchmark may load it. It shares no code, header, table or constant
// with the CUDA library, and it never reads anything the CUDA library produced.
//
// Sources (web pages of the NVIDIA/Model-Optimizer pull requests on the method):
//   [F]  "GDN state/W QAT foundation" (#2497), section "What does this PR do?":
//        state QDQ at 64-token boundaries, one scale per full-key x 64-value-column
//        tile per sequence and head, scale = amax / 448 (1 for an all-zero tile), E4M3
//        (num_bits (4,3)); independent dynamic FP8 QDQ of the WY-transformed W.
//   [D]  "Torch GDN/KDA decode QAT with INT8 recurrent state" (#2519), section
//        "Megatron-Core QAT/QAD workflow", step 3: per decode token the stored state is
//        loaded and updated, the output comes from that updated state before any
//        quantization, and the state is QDQ'd before it is written back for the next token.
//   [K]  "Add KDA prefill numerical emulation for QAT" (#2506), section "What does
//        this PR do?": KDA has per-key-channel retention; causal pairwise
//        exponentials come from prefix differences of the log decay.
//   [R]  "Add experimental GDN/KDA decode and replay QAT" (#2509), section "What does
//        this PR do?": per-token FP8 state writes in decode.
//   [I]  "Torch GDN/KDA decode QAT with INT8 recurrent state" (#2519): its summary names an
//        INT8 state codec whose scales cover 32-value blocks; the shipped recipe
//        linear_attention_state_int8_block32_dynamic ("Megatron-Core QAT/QAD workflow" step 1
//        and "Usage"); the INT8 state is signed; and "Add experimental GDN/KDA decode and replay
//        QAT" tests state and value tails at codec block sizes 32 and 128. Read as: a block is 32
//        consecutive value columns of one key row of the state (the last block of a row may be
//        narrower); scale = amax / 127 with the same zero guard as the E4M3 tiles; code = the
//        signed integer nearest x / scale (ties to even), kept within [-127, 127].
//   [H]  "Torch GDN/KDA decode QAT with INT8 recurrent state" (#2519), section
//        "Megatron-Core QAT/QAD workflow", steps 2-3 and the "Ordinary state-QDQ path"
//        flowchart: a sequence's first prefill_lengths tokens run as chunked prefill whose
//        state is never quantized inside the prefix; if any tokens are left, the state is
//        QDQ'd once when the prefix hands over, and each remaining token (teacher forced, the
//        sequence's own tokens) is a decode step that QDQs the state before storing it.
// The pages name GatedDeltaNet but never print its recurrence. The oracle uses the
// standard gated delta rule for a state S in R^{dk x dv}:
//     S_t = a_t S_{t-1} + b_t k_t (v_t - a_t S_{t-1}^T k_t)^T,   o_t = S_t^T q_t,
// with a_t = exp(g_t) (KDA: S_{t-1} rows scaled by exp(g_t[c]) per key channel c).
//
// Functions (all extern "C", row-major; fp32 inputs widened to fp64, h0 given in fp64):
//   oracle_e4m3_rne          E4M3 round-to-nearest-even with saturation
//   oracle_tile_qdq_f32      fp32 tile QDQ, bit-for-bit definition of the standalone op
//   oracle_tile_qdq_f64      the same steps in fp64 (used inside the fp64 oracles)
//   oracle_gdn_recurrent     O1: token-by-token recurrence (the definition)
//   oracle_gdn_chunked       O2: chunked / WY form (the only form in which W QDQ exists)
//   oracle_gdn_decode        single-token decode steps with per-token state QDQ
//   oracle_gdn_prefill_decode  [H]: chunked prefix (no state QDQ), QDQ at the handoff,
//                            recurrent suffix with per-token state QDQ
//   oracle_int8_block_qdq_f32 / _f64  [I]: the INT8 block codec (fp32: bit-for-bit definition
//                            of the standalone op)
// The state_qdq argument of the prefill / decode functions selects the state codec: 0 off,
// 1 E4M3 tiles [F], 2 INT8 blocks of 32 value columns [I].
// Every function is pinned by tests/test_oracle_*.py against closed forms, invariants,
// hand-worked examples and brute force.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// E4M3 (OCP FP8 "fn" variant: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
// bits, no infinities, largest finite value 1.75 * 2^8 = 448, smallest subnormal 2^-9).
// Rounding: to nearest, ties to even mantissa; magnitudes past the largest finite value
// saturate to +-448 ("satfinite"). Written from the format definition.
// ---------------------------------------------------------------------------
const double kE4M3Max = 448.0;

double e4m3_rne_sat(double y) {
  if (std::isnan(y)) return y;
  const double a = std::fabs(y);
  if (a == 0.0) return std::copysign(0.0, y);
  if (a >= kE4M3Max) return std::copysign(kE4M3Max, y);
  int e = 0;
  std::frexp(a, &e);          // a = m * 2^e with m in [0.5, 1): leading bit is 2^(e-1)
  int lead = e - 1;
  if (lead < -6) lead = -6;   // subnormals share the spacing of the lowest normal binade
  const double quantum = std::ldexp(1.0, lead - 3);   // 3 mantissa bits
  double c = std::nearbyint(a / quantum) * quantum;   // default mode: nearest, ties to even
  if (c > kE4M3Max) c = kE4M3Max;
  return std::copysign(c, y);
}

// One QDQ tile: rows x cols elements at x[r * ld + j]. Steps as stated on [F]:
// amax over the tile, scale = amax / 448 (zero guard: 0 -> 1), x <- E4M3(x / scale) * scale.
template <typename R>
R qdq_tile(R* x, int64_t ld, int rows, int cols) {
  R amax = 0;
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < cols; ++j) amax = std::max(amax, (R)std::fabs(x[r * ld + j]));
  R s = amax / (R)448;
  if (s == (R)0) s = (R)1;
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < cols; ++j) {
      R y = x[r * ld + j] / s;
      R c = (R)e4m3_rne_sat((double)y);   // exact: c is an E4M3 value, representable in R
      x[r * ld + j] = c * s;
    }
  return s;
}

// INT8 [I]: round to the nearest integer (ties to even), kept within [-127, 127].
double int8_rne_sat(double y) {
  if (std::isnan(y)) return y;
  const double c = std::nearbyint(y);   // default mode: nearest, ties to even
  return std::min(127.0, std::max(-127.0, c));
}

// One INT8 block: n consecutive elements; scale = amax / 127 (zero guard: 0 -> 1),
// x <- INT8(x / scale) * scale.
template <typename R>
R qdq_int8_block(R* x, int n) {
  R amax = 0;
  for (int j = 0; j < n; ++j) amax = std::max(amax, (R)std::fabs(x[j]));
  R s = amax / (R)127;
  if (s == (R)0) s = (R)1;
  for (int j = 0; j < n; ++j) {
    R y = x[j] / s;
    R c = (R)int8_rne_sat((double)y);   // exact: an integer of magnitude <= 127
    x[j] = c * s;
  }
  return s;
}

// State QDQ of one (sequence, head) state S[dk][dv]. Codec 1 [F]: one E4M3 tile per 64 value
// columns spanning all dk key rows. Codec 2 [I]: one INT8 block per key row and 32 value columns.
const int kStateTileCols = 64;
const int kInt8BlockCols = 32;
void qdq_state(double* S, int dk, int dv, int codec) {
  if (codec == 2) {
    for (int c = 0; c < dk; ++c)
      for (int j0 = 0; j0 < dv; j0 += kInt8BlockCols)
        qdq_int8_block<double>(S + (size_t)c * dv + j0, std::min(kInt8BlockCols, dv - j0));
    return;
  }
  for (int j0 = 0; j0 < dv; j0 += kStateTileCols)
    qdq_tile<double>(S + j0, dv, dk, std::min(kStateTileCols, dv - j0));
}

// ---------------------------------------------------------------------------
// Problem description shared by the prefill oracles.
// Layout: q, k [B, T, Hqk, dk]; v [B, T, Hv, dv]; g [B, T, Hv] (KDA: [B, T, Hv, dk]);
// beta [B, T, Hv]; h0, hT [N, Hv, dk, dv]; o [B, T, Hv, dv]. With cu_seqlens (B == 1),
// sequence n owns tokens [cu_seqlens[n], cu_seqlens[n+1]) of the packed T axis.
// GQA: v-head h reads q/k head h / (Hv / Hqk).
// ---------------------------------------------------------------------------
struct Problem {
  const float *q, *k, *v, *g, *beta;
  const double* h0;   // fp64 so that a final state can be fed back bit-for-bit
  const int32_t* cu;
  int B, T, N, Hqk, Hv, dk, dv, kda;
  double scale;
};

struct UnitRange { int64_t t0, len; };

UnitRange unit_range(const Problem& p, int n) {
  if (p.cu) return {p.cu[n], (int64_t)p.cu[n + 1] - p.cu[n]};
  return {(int64_t)n * p.T, p.T};
}

// log-decay of token tok (global packed index), head h, key channel c
double logdecay(const Problem& p, int64_t tok, int h, int c) {
  if (p.kda) return (double)p.g[(tok * p.Hv + h) * p.dk + c];
  return (double)p.g[tok * p.Hv + h];
}

void load_h0(const Problem& p, int n, int h, double* S) {
  const int64_t sz = (int64_t)p.dk * p.dv;
  if (p.h0) {
    const double* src = p.h0 + ((int64_t)n * p.Hv + h) * sz;
    std::copy(src, src + sz, S);
  } else {
    std::fill(S, S + sz, 0.0);
  }
}

// One token of the recurrence for head h at packed token index tok, on the state S
// (steps 1-5; the caller decides on the QDQ of step 6).
void recurrent_step(const Problem& p, int64_t tok, int h, double* S, double* o) {
  const int dk = p.dk, dv = p.dv, hq = h / (p.Hv / p.Hqk);
  std::vector<double> d(dv), kv(dk), qv(dk);
  for (int c = 0; c < dk; ++c) {
    kv[c] = (double)p.k[(tok * p.Hqk + hq) * dk + c];
    qv[c] = (double)p.q[(tok * p.Hqk + hq) * dk + c];
  }
  const double b = (double)p.beta[tok * p.Hv + h];
  // 1. S' = alpha S (KDA: row c scaled by alpha[c])
  for (int c = 0; c < dk; ++c) {
    const double a = std::exp(logdecay(p, tok, h, c));
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
  }
  // 2. p = S'^T k ; 3. delta = beta (v - p)
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * kv[c];
    d[j] = b * ((double)p.v[(tok * p.Hv + h) * dv + j] - acc);
  }
  // 4. S = S' + k delta^T
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += kv[c] * d[j];
  // 5. o = scale * S^T q  (from the updated, not yet quantized state)
  if (o) {
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qv[c];
      o[(tok * p.Hv + h) * dv + j] = p.scale * acc;
    }
  }
}

// O1: the recurrence itself, one token at a time. QDQ of S after every token whose
// sequence-local count is a multiple of qdq_period (64 for prefill per [F]).
void recurrent_unit(const Problem& p, int n, int h, int state_qdq, int qdq_period,
                    double* o, double* hT) {
  const int dk = p.dk, dv = p.dv;
  const UnitRange u = unit_range(p, n);
  std::vector<double> S((size_t)dk * dv);
  load_h0(p, n, h, S.data());
  for (int64_t t = 0; t < u.len; ++t) {
    recurrent_step(p, u.t0 + t, h, S.data(), o);
    // 6. state QDQ at the boundary
    if (state_qdq && ((t + 1) % qdq_period) == 0) qdq_state(S.data(), dk, dv, state_qdq);
  }
  if (hT) std::copy(S.begin(), S.end(), hT + ((int64_t)n * p.Hv + h) * (int64_t)dk * dv);
}

// O2: chunked / WY form with chunk length C (the pages fix C = 64; other C are for the
// equivalence pin). Per chunk of L tokens entering with state S0:
//   gam_r = sum_{j<=r} g_j                   (KDA: per key channel)
//   A[r][i] = beta_r * sum_c k_r[c] k_i[c] exp(gam_r[c] - gam_i[c]),  i < r
//   Tm = (I + A)^{-1}                        (forward substitution, row by row)
//   W = Tm (beta * exp(gam) * K),  U = Tm (beta * V)
//   W <- QDQ(W) as one L x dk tile           (when w_qdq)
//   Delta = U - W S0
//   o_r = scale [ sum_c q_r[c] exp(gam_r[c]) S0[c,:] + sum_{i<=r} P[r][i] Delta_i ],
//         P[r][i] = sum_c q_r[c] k_i[c] exp(gam_r[c] - gam_i[c])
//   S1[c,:] = exp(gam_L[c]) S0[c,:] + sum_i k_i[c] exp(gam_L[c] - gam_i[c]) Delta_i
//   S1 <- QDQ(S1) when the chunk ends on a 64-token boundary of its sequence.
// Unrolling the recurrence over a chunk gives S_r = Gam_r S0 + sum_{i<=r} (Gam_r/Gam_i)
// k_i d_i^T; putting that into d_r = b_r (v_r - a_r S_{r-1}^T k_r) gives
// (I + A) Delta = beta V - (beta Gam K) S0, i.e. Delta = U - W S0.
// Runs the chunks of tokens [u.t0, u.t0 + u.len) of head h on the state S (in / out); chunk
// and boundary positions count from u.t0, the sequence's first token.
void chunked_range(const Problem& p, UnitRange u, int h, int C, int state_qdq, int w_qdq,
                   double* o, std::vector<double>& S) {
  const int dk = p.dk, dv = p.dv, hq = h / (p.Hv / p.Hqk);
  std::vector<double> S1((size_t)dk * dv);
  std::vector<double> K((size_t)C * dk), Q((size_t)C * dk), V((size_t)C * dv), bt(C);
  std::vector<double> gam((size_t)C * dk), A((size_t)C * C), Tm((size_t)C * C);
  std::vector<double> X((size_t)C * dk), W((size_t)C * dk), U((size_t)C * dv), Dl((size_t)C * dv);
  for (int64_t c0 = 0; c0 < u.len; c0 += C) {
    const int L = (int)std::min<int64_t>(C, u.len - c0);
    for (int r = 0; r < L; ++r) {
      const int64_t tok = u.t0 + c0 + r;
      for (int c = 0; c < dk; ++c) {
        K[(size_t)r * dk + c] = (double)p.k[(tok * p.Hqk + hq) * dk + c];
        Q[(size_t)r * dk + c] = (double)p.q[(tok * p.Hqk + hq) * dk + c];
        const double prev = r ? gam[(size_t)(r - 1) * dk + c] : 0.0;
        gam[(size_t)r * dk + c] = prev + logdecay(p, tok, h, c);
      }
      for (int j = 0; j < dv; ++j) V[(size_t)r * dv + j] = (double)p.v[(tok * p.Hv + h) * dv + j];
      bt[r] = (double)p.beta[tok * p.Hv + h];
    }
    // A (strictly lower)
    for (int r = 0; r < L; ++r)
      for (int i = 0; i < L; ++i) {
        double acc = 0.0;
        if (i < r)
          for (int c = 0; c < dk; ++c)
            acc += K[(size_t)r * dk + c] * K[(size_t)i * dk + c] *
                   std::exp(gam[(size_t)r * dk + c] - gam[(size_t)i * dk + c]);
        A[(size_t)r * C + i] = bt[r] * acc;
      }
    // Tm = (I + A)^{-1}: row r of Tm is e_r - sum_{i<r} A[r][i] * (row i of Tm)
    for (int r = 0; r < L; ++r)
      for (int j = 0; j < L; ++j) {
        double acc = (r == j) ? 1.0 : 0.0;
        for (int i = 0; i < r; ++i) acc -= A[(size_t)r * C + i] * Tm[(size_t)i * C + j];
        Tm[(size_t)r * C + j] = acc;
      }
    // W = Tm X with X = beta * exp(gam) * K ;  U = Tm (beta * V)
    for (int i = 0; i < L; ++i)
      for (int c = 0; c < dk; ++c)
        X[(size_t)i * dk + c] = bt[i] * std::exp(gam[(size_t)i * dk + c]) * K[(size_t)i * dk + c];
    for (int r = 0; r < L; ++r) {
      for (int c = 0; c < dk; ++c) {
        double acc = 0.0;
        for (int i = 0; i < L; ++i) acc += Tm[(size_t)r * C + i] * X[(size_t)i * dk + c];
        W[(size_t)r * dk + c] = acc;
      }
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < L; ++i) acc += Tm[(size_t)r * C + i] * bt[i] * V[(size_t)i * dv + j];
        U[(size_t)r * dv + j] = acc;
      }
    }
    if (w_qdq) qdq_tile<double>(W.data(), dk, L, dk);
    // Delta = U - W S0
    for (int r = 0; r < L; ++r)
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += W[(size_t)r * dk + c] * S[(size_t)c * dv + j];
        Dl[(size_t)r * dv + j] = U[(size_t)r * dv + j] - acc;
      }
    // outputs (the row factors qg[c] = q_r[c] exp(gam_r[c]) and P[r][i] do not depend on the
    // value column j, so they are formed once per row)
    if (o) {
      for (int r = 0; r < L; ++r) {
        const int64_t tok = u.t0 + c0 + r;
        for (int c = 0; c < dk; ++c) X[c] = Q[(size_t)r * dk + c] * std::exp(gam[(size_t)r * dk + c]);
        for (int i = 0; i <= r; ++i) {
          double pri = 0.0;
          for (int c = 0; c < dk; ++c)
            pri += Q[(size_t)r * dk + c] * K[(size_t)i * dk + c] *
                   std::exp(gam[(size_t)r * dk + c] - gam[(size_t)i * dk + c]);
          A[i] = pri;   // A is free once Tm is formed: row r of P
        }
        for (int j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int c = 0; c < dk; ++c) acc += X[c] * S[(size_t)c * dv + j];
          for (int i = 0; i <= r; ++i) acc += A[i] * Dl[(size_t)i * dv + j];
          o[(tok * p.Hv + h) * dv + j] = p.scale * acc;
        }
      }
    }
    // state carried to the next chunk
    for (int c = 0; c < dk; ++c) {
      const double gl = gam[(size_t)(L - 1) * dk + c];
      for (int i = 0; i < L; ++i) X[i] = K[(size_t)i * dk + c] * std::exp(gl - gam[(size_t)i * dk + c]);
      for (int j = 0; j < dv; ++j) {
        double acc = std::exp(gl) * S[(size_t)c * dv + j];
        for (int i = 0; i < L; ++i) acc += X[i] * Dl[(size_t)i * dv + j];
        S1[(size_t)c * dv + j] = acc;
      }
    }
    S.swap(S1);
    if (state_qdq && ((c0 + L) % 64) == 0) qdq_state(S.data(), dk, dv, state_qdq);
  }
}

void chunked_unit(const Problem& p, int n, int h, int C, int state_qdq, int w_qdq,
                  double* o, double* hT) {
  std::vector<double> S((size_t)p.dk * p.dv);
  load_h0(p, n, h, S.data());
  chunked_range(p, unit_range(p, n), h, C, state_qdq, w_qdq, o, S);
  if (hT) std::copy(S.begin(), S.end(), hT + ((int64_t)n * p.Hv + h) * (int64_t)p.dk * p.dv);
}

// [H] for one (sequence, head): the first P tokens as chunked prefill (chunk 64) with no
// state QDQ (W QDQ as asked), then -- if tokens remain -- QDQ of the handed-off state and
// the remaining tokens one by one, each followed by a state QDQ (state_qdq on).
void prefill_decode_unit(const Problem& p, int n, int h, int64_t P, int state_qdq, int w_qdq,
                         double* o, double* hT) {
  const UnitRange u = unit_range(p, n);
  std::vector<double> S((size_t)p.dk * p.dv);
  load_h0(p, n, h, S.data());
  chunked_range(p, UnitRange{u.t0, P}, h, 64, 0, w_qdq, o, S);
  if (P < u.len) {
    if (state_qdq) qdq_state(S.data(), p.dk, p.dv, state_qdq);
    for (int64_t t = P; t < u.len; ++t) {
      recurrent_step(p, u.t0 + t, h, S.data(), o);
      if (state_qdq) qdq_state(S.data(), p.dk, p.dv, state_qdq);
    }
  }
  if (hT) std::copy(S.begin(), S.end(), hT + ((int64_t)n * p.Hv + h) * (int64_t)p.dk * p.dv);
}

// Run fn(n, h) for every selected (n, h) unit on `threads` std::threads.
template <typename F>
void for_units(int N, int Hv, const uint8_t* mask, int threads, F fn) {
  const int total = N * Hv;
  std::atomic<int> next(0);
  auto worker = [&]() {
    for (int i = next++; i < total; i = next++)
      if (!mask || mask[i]) fn(i / Hv, i % Hv);
  };
  threads = std::max(1, std::min(threads, total));
  std::vector<std::thread> pool;
  for (int t = 1; t < threads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

int check_problem(const Problem& p) {
  if (!p.q || !p.k || !p.v || !p.g || !p.beta) return 1;
  if (p.Hqk <= 0 || p.Hv <= 0 || p.Hv % p.Hqk != 0 || p.dk <= 0 || p.dv <= 0) return 1;
  if (p.cu) {
    if (p.B != 1 || p.N <= 0 || p.cu[0] != 0 || p.cu[p.N] != p.T) return 1;
    for (int n = 0; n < p.N; ++n)
      if (p.cu[n + 1] < p.cu[n]) return 1;
  } else if (p.N != p.B) {
    return 1;
  }
  return 0;
}

}  // namespace

extern "C" {

double oracle_e4m3_rne(double y) { return e4m3_rne_sat(y); }

// Standalone fp32 tile QDQ. x, y: [lead, rows, cols] fp32 (y may equal x); one tile is all
// `rows` x `tile_cols` columns (the last tile of a row block may be narrower) of one leading
// index. scales (nullable): [lead, ceil(cols / tile_cols)] fp32. Every step in fp32 with
// IEEE round-to-nearest: amax, s = amax / 448 (0 -> 1), y = x / s, E4M3, c * s.
int oracle_tile_qdq_f32(const float* x, float* y, float* scales, int64_t lead, int rows,
                        int cols, int tile_cols) {
  if (!x || !y || lead < 0 || rows < 0 || cols < 0 || tile_cols <= 0) return 1;
  const int ntiles = (cols + tile_cols - 1) / tile_cols;
  const int64_t mat = (int64_t)rows * cols;
  if (y != x) std::memcpy(y, x, sizeof(float) * (size_t)(lead * mat));
  for (int64_t l = 0; l < lead; ++l)
    for (int t = 0; t < ntiles; ++t) {
      const int j0 = t * tile_cols;
      const float s = qdq_tile<float>(y + l * mat + j0, cols, rows, std::min(tile_cols, cols - j0));
      if (scales) scales[l * ntiles + t] = s;
    }
  return 0;
}

// The same tile QDQ in fp64 (the arithmetic used inside the fp64 oracles).
int oracle_tile_qdq_f64(double* x, double* scales, int64_t lead, int rows, int cols,
                        int tile_cols) {
  if (!x || lead < 0 || rows < 0 || cols < 0 || tile_cols <= 0) return 1;
  const int ntiles = (cols + tile_cols - 1) / tile_cols;
  const int64_t mat = (int64_t)rows * cols;
  for (int64_t l = 0; l < lead; ++l)
    for (int t = 0; t < ntiles; ++t) {
      const int j0 = t * tile_cols;
      const double s = qdq_tile<double>(x + l * mat + j0, cols, rows, std::min(tile_cols, cols - j0));
      if (scales) scales[l * ntiles + t] = s;
    }
  return 0;
}

// O1. Outputs o [B, T, Hv, dv] and hT [N, Hv, dk, dv] in fp64 (either may be null);
// unit_mask [N * Hv] (nullable) selects the (n, h) units to compute.
// INT8 block codec [I], every step in fp32 with IEEE round-to-nearest: per block of
// block_cols consecutive columns of a row (the last block of a row may be narrower),
// amax = max |x|, s = amax / 127 (s == 0 -> 1), c = nearest integer to x / s (ties to even)
// within [-127, 127], y = c * s. x, y: [rows, cols] fp32 (y may equal x); scales (nullable):
// [rows, ceil(cols / block_cols)].
int oracle_int8_block_qdq_f32(const float* x, float* y, float* scales, int64_t rows, int cols, int block_cols) {
  if (!x || !y || rows < 0 || cols < 0 || block_cols <= 0) return 1;
  const int nb = (cols + block_cols - 1) / block_cols;
  if (y != x) std::memcpy(y, x, sizeof(float) * (size_t)(rows * cols));
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b) {
      const float s = qdq_int8_block<float>(y + r * cols + b * block_cols, std::min(block_cols, cols - b * block_cols));
      if (scales) scales[r * nb + b] = s;
    }
  return 0;
}

// The same codec in fp64 (the arithmetic used inside the fp64 oracles).
int oracle_int8_block_qdq_f64(double* x, double* scales, int64_t rows, int cols, int block_cols) {
  if (!x || rows < 0 || cols < 0 || block_cols <= 0) return 1;
  const int nb = (cols + block_cols - 1) / block_cols;
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b) {
      const double s = qdq_int8_block<double>(x + r * cols + b * block_cols, std::min(block_cols, cols - b * block_cols));
      if (scales) scales[r * nb + b] = s;
    }
  return 0;
}

int oracle_gdn_recurrent(const float* q, const float* k, const float* v, const float* g,
                         const float* beta, const double* h0, const int32_t* cu_seqlens,
                         int B, int T, int N, int Hqk, int Hv, int dk, int dv, int kda,
                         int state_qdq, int qdq_period, double scale,
                         const uint8_t* unit_mask, int threads, double* o, double* hT) {
  Problem p{q, k, v, g, beta, h0, cu_seqlens, B, T, N, Hqk, Hv, dk, dv, kda, scale};
  if (check_problem(p) || qdq_period <= 0 || state_qdq < 0 || state_qdq > 2) return 1;
  for_units(N, Hv, unit_mask, threads, [&](int n, int h) {
    recurrent_unit(p, n, h, state_qdq, qdq_period, o, hT);
  });
  return 0;
}

// O2. Same arguments as O1 plus the chunk length and the W QDQ switch.
int oracle_gdn_chunked(const float* q, const float* k, const float* v, const float* g,
                       const float* beta, const double* h0, const int32_t* cu_seqlens,
                       int B, int T, int N, int Hqk, int Hv, int dk, int dv, int kda,
                       int chunk, int state_qdq, int w_qdq, double scale,
                       const uint8_t* unit_mask, int threads, double* o, double* hT) {
  Problem p{q, k, v, g, beta, h0, cu_seqlens, B, T, N, Hqk, Hv, dk, dv, kda, scale};
  if (check_problem(p) || chunk <= 0 || state_qdq < 0 || state_qdq > 2) return 1;
  for_units(N, Hv, unit_mask, threads, [&](int n, int h) {
    chunked_unit(p, n, h, chunk, state_qdq, w_qdq, o, hT);
  });
  return 0;
}

// [H]. Same arguments as O2 (chunk fixed at 64) plus prefill_lengths [N]: 0 <= P_n <= L_n.
int oracle_gdn_prefill_decode(const float* q, const float* k, const float* v, const float* g,
                              const float* beta, const double* h0, const int32_t* cu_seqlens,
                              const int32_t* prefill_lengths, int B, int T, int N, int Hqk, int Hv,
                              int dk, int dv, int kda, int state_qdq, int w_qdq, double scale,
                              const uint8_t* unit_mask, int threads, double* o, double* hT) {
  Problem p{q, k, v, g, beta, h0, cu_seqlens, B, T, N, Hqk, Hv, dk, dv, kda, scale};
  if (check_problem(p) || !prefill_lengths || state_qdq < 0 || state_qdq > 2) return 1;
  for (int n = 0; n < N; ++n)
    if (prefill_lengths[n] < 0 || prefill_lengths[n] > unit_range(p, n).len) return 1;
  for_units(N, Hv, unit_mask, threads, [&](int n, int h) {
    prefill_decode_unit(p, n, h, prefill_lengths[n], state_qdq, w_qdq, o, hT);
  });
  return 0;
}

// Decode: `steps` single-token steps for N sequences. Inputs per step s:
// q, k [steps, N, Hqk, dk]; v [steps, N, Hv, dv]; g [steps, N, Hv] (KDA [.., dk]);
// beta [steps, N, Hv]. state [N, Hv, dk, dv] fp64 in/out; o [steps, N, Hv, dv] fp64.
// Per token, in the order of [D]: load the stored state, update it, take o from the updated
// state, then QDQ it (when state_qdq) and store it.
int oracle_gdn_decode(const float* q, const float* k, const float* v, const float* g,
                      const float* beta, int steps, int N, int Hqk, int Hv, int dk, int dv,
                      int kda, int state_qdq, double scale, const uint8_t* unit_mask,
                      int threads, double* state, double* o) {
  if (!q || !k || !v || !g || !beta || !state || steps < 0 || N < 0 || state_qdq < 0 || state_qdq > 2) return 1;
  if (Hqk <= 0 || Hv <= 0 || Hv % Hqk != 0 || dk <= 0 || dv <= 0) return 1;
  const int G = Hv / Hqk;
  for_units(N, Hv, unit_mask, threads, [&](int n, int h) {
    const int hq = h / G;
    double* S = state + ((int64_t)n * Hv + h) * (int64_t)dk * dv;
    std::vector<double> d(dv);
    for (int s = 0; s < steps; ++s) {
      const int64_t row = (int64_t)s * N + n;   // token index in the [steps, N] grid
      const float* kt = k + (row * Hqk + hq) * dk;
      const float* qt = q + (row * Hqk + hq) * dk;
      const float* vt = v + (row * Hv + h) * dv;
      const double b = (double)beta[row * Hv + h];
      for (int c = 0; c < dk; ++c) {
        const double a = std::exp((double)(kda ? g[(row * Hv + h) * dk + c] : g[row * Hv + h]));
        for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
      }
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * (double)kt[c];
        d[j] = b * ((double)vt[j] - acc);
      }
      for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += (double)kt[c] * d[j];
      if (o) {
        for (int j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * (double)qt[c];
          o[(row * Hv + h) * dv + j] = scale * acc;
        }
      }
      if (state_qdq) qdq_state(S, dk, dv, state_qdq);
    }
  });
  return 0;
}

}  // extern "C"
