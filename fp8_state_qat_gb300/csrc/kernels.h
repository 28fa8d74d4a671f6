// kernels.h -- internal launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdnqat.h"

namespace gdn {

// The current device is an sm_103 GPU (cached per device ordinal below 64); checked by every
// entry point before it enqueues anything.
gdn_status check_device();
// The status word of the array behind gdn_chunk_fwd_noalloc on the current device (synchronous).
gdn_status noalloc_status_word(int* word);

struct ChunkProblem {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;   // device cu_seqlens or null
  float* o;
  float* hT;
  int B, T, N, Hqk, Hv, dk, dv;
  float scale;
  int state_qdq, w_qdq, kda;
  const int32_t* cu_host = nullptr;   // host copy of cu_seqlens (when known): orders the chain CTAs
  // Tokens of each sequence this pass runs, from the sequence's first token (device [N] and its
  // host copy), or null for whole sequences: the prefill part of a prefill -> decode handoff.
  const int32_t* lens = nullptr;
  const int32_t* lens_host = nullptr;
  // Scales of the final state's QDQ, or null: E4M3 (state_qdq 1) fp32 [N, Hv, dv / 64] per tile,
  // INT8 (state_qdq 2) fp32 [N, Hv, dk, dv / 32] per block; 0 where the final state was not QDQ'd.
  float* state_scales = nullptr;
};

cudaError_t launch_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int rows, int cols,
                            int tile_cols, cudaStream_t stream);
// INT8 block QDQ: x, y [rows, cols] fp32, one block = block_cols consecutive columns of a row.
cudaError_t launch_int8_block_qdq(const float* x, float* y, float* scales, int64_t rows, int cols, int block_cols,
                                  cudaStream_t stream);

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, float* o, int N, int Hqk, int Hv, int dk, int dv, float scale,
                          int state_qdq, int kda, cudaStream_t stream);

// Fused tensor-core chunked forward (tcgen05 + TMA), dk = 128, GDN. status: device int,
// set to nonzero when a bounded wait gives up.
bool chunk_tc_supported(const ChunkProblem& p);
cudaError_t launch_chunk_tc(const ChunkProblem& p, int* status, cudaStream_t stream);

// TMA descriptor of a head-last bf16 tensor [tokens, heads, D] with 64 x 1 x box_tokens boxes
// (128-byte swizzle). Host only; false when the driver entry point is unavailable.
bool make_bf16_map(CUtensorMap* map, const void* base, int D, int heads, int64_t tokens, int box_tokens = 64);
// TMA descriptor of a bf16 matrix [rows][64] with 64 x box_rows boxes (128-byte swizzle).
bool make_bf16_rows_map(CUtensorMap* map, const void* base, int64_t rows, int box_rows);
// TMA descriptor of a head-last fp32 output [tokens, heads, D] with 32 x 1 x 64 boxes (128-byte swizzle).
bool make_f32_out_map(CUtensorMap* map, void* base, int D, int heads, int64_t tokens);

// ---- split tensor-core path: a parallel prep kernel, then the state-carrying chain kernel ----
// Work items are (slot, v-head); slot(n, c) = floor(cu[n] / 64) + n + c for chunk c of sequence n
// (cu[n] = n T without cu_seqlens). The slots of different sequences never collide, and there
// are at most floor(tokens / 64) + N of them. Per item the prep kernel stores, in the workspace:
//   W    bf16 [2 key blocks][64 r][64 c]: the chunk's W, key columns 0-63 then 64-127 -- E4M3
//        codes (exact in bf16) with W QDQ, else the bf16 hi part followed by the lo part
//        ([2][2][64][64]);
//   T''  bf16 [128][64 i]: hi and lo parts of T diag(beta) (U = T'' V in the chain), rows
//        interleaved in 16-row groups: row 32 g + s is hi row 16 g + s, row 32 g + 16 + s lo row 16 g + s;
//   P    bf16 [128][64 i]: hi and lo parts of exp(gam_r - gam_i) (q_r . k_i), i <= r < L, rows
//        interleaved the same way;
//   vec  fp32 [256]: gam [64], Gam = exp(gam) [64], exp(gam_63 - gam) [64], W scale (index 192).
struct SplitLayout {
  int64_t slots, items;
  size_t wt_item_bytes;            // W: 16 KB with W QDQ, 32 KB without
  size_t off_wt, off_tt, off_p, off_vec;  // byte offsets inside the workspace
  size_t off_order;                // N int32: sequences by decreasing length (varlen chain order)
  size_t total;                    // workspace bytes, status word included
};
constexpr size_t kStatusBytes = 256;   // the device status word, padded to one line
bool chunk_split_supported(const ChunkProblem& p);
SplitLayout chunk_split_layout(const ChunkProblem& p);
// ws: the workspace (status word at offset 0), ws_bytes >= chunk_split_layout(p).total.
cudaError_t launch_chunk_split(const ChunkProblem& p, void* ws, cudaStream_t stream);
// Chain CTAs of the longest sequences first: with more (sequence, head, slab) chains than SMs the
// makespan is then close to total work / SMs. Writes the order into ws + off_order (N int32,
// staged from host memory) and returns its device address, or null for one sequence, dense
// batches of whole sequences (equal lengths) or no host copy of the lengths.
const int32_t* stage_chain_order(const ChunkProblem& p, unsigned char* ws, size_t off_order, cudaStream_t stream,
                                 cudaError_t* err);

// ---- the same split for KDA (per-key-channel decay), dk = 128 ----
// Per item the KDA prep kernel stores W^T, T'' as for GDN, plus
//   P    bf16 [2][64 r][64 i]: hi | lo of sum_c q_r[c] k_i[c] exp(gam_r[c] - gam_i[c]), i <= r;
//   Qd   bf16 [2][2][64 r][64 c]: hi | lo of q_r[c] exp(gam_r[c]), key blocks c < 64 | c >= 64;
//   Kd   bf16 [2][2][64 i][64 c]: hi | lo of k_i[c] exp(gam_63[c] - gam_i[c]), same blocks;
//   vec  fp32 [256]: exp(gam_63[c]) for c < 128, W scale at index 192.
struct KdaLayout {
  int64_t slots, items;
  size_t wt_item_bytes;
  size_t off_wt, off_tt, off_p, off_qd, off_kd, off_vec, off_order;
  size_t total;
};
bool kda_split_supported(const ChunkProblem& p);
KdaLayout kda_split_layout(const ChunkProblem& p);
cudaError_t launch_kda_split(const ChunkProblem& p, void* ws, cudaStream_t stream);

// Per-CTA fp32 chunked forward on CUDA cores: one CTA per (sequence, head, 64-column
// value slab). Used for shapes and variants the tensor-core path does not take.
cudaError_t launch_chunk_simt(const ChunkProblem& p, cudaStream_t stream);

// The decode part of a prefill -> decode handoff: for every (sequence, head) whose sequence has
// tokens past its prefill length P_n, read the state from hT, QDQ it (state_qdq), then run the
// tokens [P_n, L_n) one by one as decode steps (teacher forced: q, k, v, g, beta of those tokens;
// o of those tokens written), each followed by a state QDQ (state_qdq), and store the state back
// into hT. plens: device [N]; the state stays in registers across the tokens.
cudaError_t launch_handoff_suffix(const ChunkProblem& p, const int32_t* plens, cudaStream_t stream);

// ---- backward with straight-through state QDQ (CUDA cores, recurrent form) ----
struct BwdGrads {
  const float* dout;   // [tokens, Hv, dv]
  const float* dhT;    // [N, Hv, dk, dv] or null (zero)
  float* dq;           // [tokens, Hqk, dk]
  float* dk;           // [tokens, Hqk, dk]
  float* dv;           // [tokens, Hv, dv]
  float* dg;           // [tokens, Hv] (KDA [tokens, Hv, dk])
  float* dbeta;        // [tokens, Hv]
  float* dh0;          // [N, Hv, dk, dv] or null
};
// workspace: status word, the state entering every chunk (per chunk slot and v-head), one
// 64-state slab scratch per CTA, and the per-slab, per-v-head dq, dk, db, dg before their sums
struct BwdLayout {
  size_t off_ckpt, off_scratch, off_part_q, off_part_k, off_part_b, off_part_g, total;
};
BwdLayout chunk_bwd_layout(const ChunkProblem& p);
cudaError_t launch_chunk_bwd(const ChunkProblem& p, const BwdGrads& gr, void* ws, cudaStream_t stream);

}  // namespace gdn
