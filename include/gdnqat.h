/* gdnqat.h -- C ABI of the GB300 (sm_103a) chunked gated-delta-rule forward with dynamic
 * FP8 E4M3 fake quantize-dequantize (QDQ) of the recurrent state and of the WY operand W.
 *
 * Sources (pages of the NVIDIA/Model-Optimizer pull requests on the method):
 *  [F] "GDN state/W QAT foundation", "What does this PR do?": the fused path uses chunk
 *      size 64; state QDQ at each 64-token boundary with amax recomputed over each
 *      full-key x 64-value-column tile, per sequence and head, scale = amax / 448 (1 for an
 *      all-zero tile); a separate dynamic FP8 QDQ of the WY-transformed W; quantizers start
 *      disabled; a supplied-scale QDQ helper; errors are raised before any launch.
 *  [D] "Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD
 *      workflow", step 3: per decode token the stored state is loaded and updated, the
 *      output is taken from that updated (not yet quantized) state, and the state is QDQ'd
 *      before it is written back; the stored state keeps a floating-point type.
 *  [K] "Add KDA prefill numerical emulation for QAT", "What does this PR do?": KDA uses
 *      per-key-channel retention, with causal pairwise decays from prefix differences.
 *  [R] "Add experimental GDN/KDA decode and replay QAT", "What does this PR do?":
 *      per-token FP8 state writes.
 *  [I] "Torch GDN/KDA decode QAT with INT8 recurrent state", summary: a signed INT8 state
 *      codec with one scale per 32-value block; "Add experimental GDN/KDA decode and replay QAT": codec
 *      blocks along the value columns of the state.
 *  [H] "Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD workflow",
 *      steps 2-3: chunked prefix without internal state QDQ, QDQ at the handoff, then decode
 *      tokens that QDQ the state before storing it.
 *
 * Recurrence (the pages name GatedDeltaNet but do not print it), per sequence n and
 * value head h, state S in R^{dk x dv} (row = key channel):
 *     S_t = a_t S_{t-1} + b_t k_t (v_t - a_t S_{t-1}^T k_t)^T,   o_t = scale * S_t^T q_t,
 * a_t = exp(g_t); KDA: a_t S_{t-1} becomes Diag(exp(g_t)) S_{t-1}.
 *
 * Conventions for every call
 *  - Every pointer named "device" is caller-owned device memory; the library allocates
 *    nothing and keeps no state apart from a cached per-device capability probe (and the
 *    fixed array behind gdn_chunk_fwd_noalloc).
 *  - Each call validates its arguments and the device on the host and returns a status
 *    BEFORE launching anything ([F]); a non-OK status means nothing was enqueued.
 *  - Work is enqueued on the caller's stream (NULL = legacy default stream); calls return
 *    without synchronizing. Outputs are valid once the stream reaches that point.
 *  - Layouts are head-last and contiguous: q, k [B, T, Hqk, dk] bf16; v [B, T, Hv, dv]
 *    bf16; g [B, T, Hv] fp32 (KDA [B, T, Hv, dk]); beta [B, T, Hv] fp32; states
 *    [N, Hv, dk, dv] fp32 row-major; o [B, T, Hv, dv] fp32. GQA: value head h reads
 *    q/k head h / (Hv / Hqk). Varlen: B == 1, sequence n owns tokens
 *    [cu_seqlens[n], cu_seqlens[n+1]) of the T axis.
 *  - Supported sizes: dk in {64, 128}; dv in {64, 128, 256}; chunk size 64 only ([F]).
 *    Device pointers must be 16-byte aligned.
 *  - The device must be sm_103 (GB300); the library is built for sm_103a only.
 */
#ifndef GDNQAT_H
#define GDNQAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad dims, Hv % Hqk != 0, bad cu_seqlens */
  GDN_ERR_UNSUPPORTED_ARCH = 2,     /* no CUDA device, or not sm_103 */
  GDN_ERR_UNSUPPORTED_SHAPE = 3,    /* dk / dv outside the supported set */
  GDN_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace smaller than gdn_chunk_fwd_workspace_size() */
  GDN_ERR_CUDA = 5,                 /* a CUDA runtime call or launch failed */
  GDN_ERR_DEVICE_TIMEOUT = 6        /* a kernel gave up a bounded wait (from gdn_check_device_status) */
} gdn_status;

/* Quantizer switches; all off by default, as the quantizers start disabled ([F]). */
#define GDN_FLAG_STATE_QDQ 1u  /* E4M3 QDQ of S after every 64th token of a sequence ([F]) */
#define GDN_FLAG_W_QDQ 2u      /* E4M3 QDQ of W, one scale per (sequence, head, chunk) ([F]) */
#define GDN_FLAG_KDA 4u        /* decode only: g holds one log-decay per key channel ([K]) */
#define GDN_FLAG_STATE_INT8 8u /* with GDN_FLAG_STATE_QDQ: the state QDQ uses the INT8 block codec
                                  ([I]) instead of E4M3 tiles -- one scale per key row and 32 value
                                  columns, amax / 127 with the zero guard, signed codes within
                                  +-127 (nearest, ties to even). Chunk, handoff and decode calls. */

typedef struct {
  const void* q;               /* device bf16 [B, T, Hqk, dk] */
  const void* k;               /* device bf16 [B, T, Hqk, dk] */
  const void* v;               /* device bf16 [B, T, Hv, dv] */
  const float* g;              /* device fp32 log-decay [B, T, Hv] (kda_chunk_fwd: [B, T, Hv, dk]) */
  const float* beta;           /* device fp32 [B, T, Hv] */
  const float* h0;             /* device fp32 [N, Hv, dk, dv]; NULL = zero initial state */
  const int32_t* cu_seqlens;   /* device int32 [N + 1]; NULL = dense batch (N == B) */
  const int32_t* cu_seqlens_host; /* host copy of cu_seqlens (required with it): validated before launch */
  float* o;                    /* device fp32 [B, T, Hv, dv]; must not alias any input */
  float* hT;                   /* device fp32 [N, Hv, dk, dv] or NULL; may alias h0 exactly */
  int32_t B, T, N, Hqk, Hv, dk, dv;
  float scale;                 /* multiplies o (1.0 = plain S^T q) */
  uint32_t flags;              /* GDN_FLAG_STATE_QDQ | GDN_FLAG_W_QDQ | GDN_FLAG_STATE_INT8 */
  float* state_scales;         /* device fp32 or NULL (requires GDN_FLAG_STATE_QDQ): the scales of the
                                  final state's QDQ -- E4M3 [N, Hv, dv / 64] per tile, INT8 [N, Hv, dk,
                                  dv / 32] per block; 0 where the final state was not QDQ'd (its last
                                  token was not a 64th token; a handoff without decode tokens). hT
                                  then equals code x scale, so a consumer can store hT as codes. */
} gdn_chunk_args;

/* Smallest workspace gdn_chunk_fwd / kda_chunk_fwd accept: the device status word of the
 * kernels' bounded waits, padded to one 256-byte line. */
#define GDN_CHUNK_MIN_WORKSPACE_BYTES 256

/* Bytes of device workspace for the fastest path with these arguments; 0 when the arguments
 * are invalid. For dk = 128 (GDN) that is the status word plus the staging of the two-kernel
 * path: per 64-token chunk slot and v-head, the chunk's W (transposed; E4M3 codes in bf16
 * with GDN_FLAG_W_QDQ, else bf16 hi + lo), T diag(beta) and the decay-weighted Q K^T (both
 * bf16 hi + lo) and its gate vectors -- 49 KB (65 KB without W QDQ) for each of
 * (B T / 64 + N) x Hv slots. Otherwise GDN_CHUNK_MIN_WORKSPACE_BYTES. */
size_t gdn_chunk_fwd_workspace_size(const gdn_chunk_args* args);

/* Chunked GDN forward ([F]): per 64-token chunk, decay-weighted K.K^T, WY solve (W, U),
 * optional W QDQ, state carry with state QDQ at every 64th token of each sequence; o for
 * every token and hT per (sequence, head). hT is QDQ'd when a sequence's length is a
 * positive multiple of 64 (its last token is then a 64th token). Empty sequences give
 * hT = h0. workspace: device, 256-byte aligned, at least GDN_CHUNK_MIN_WORKSPACE_BYTES;
 * its contents need no initialization. With gdn_chunk_fwd_workspace_size(args) bytes or
 * more, dk = 128 runs as two kernels (every chunk's state-independent work in parallel,
 * then the state carry); with less, as one fused kernel that does both chunk by chunk
 * (slower, same arithmetic). Returns GDN_ERR_WORKSPACE_TOO_SMALL below the minimum. */
gdn_status gdn_chunk_fwd(const gdn_chunk_args* args, void* workspace, size_t workspace_bytes,
                         gdn_stream_t stream);

/* gdn_chunk_fwd for callers that cannot allocate device memory: the pages have no
 * counterpart for this call; it exists for callers that may not call cudaMalloc (for
 * example code running inside a memory allocator's own hooks, latency-critical paths where
 * an allocation's device synchronization is not allowed, or processes whose device memory
 * is all handed to a framework's pool). Same arguments and
 * results as gdn_chunk_fwd, minus the workspace: the workspace is a 256-byte array
 * inside the library (static device memory, held by every GPU that loads the library until
 * the process exits). No cudaMalloc, cudaFree or other allocating call is made.
 *  - The device is checked first (GDN_ERR_UNSUPPORTED_ARCH on anything but sm_103); then
 *    every call looks up the array's device address (cudaGetSymbolAddress) with the
 *    device current. The first call on a device also loads the library's device code
 *    there; make that first call before any stream capture.
 *  - All calls on a device share the array (its status word is cleared at the start of
 *    each call): calls that may run at the same time on the GPU, e.g. on different
 *    streams, race on it. Serialize them, or use gdn_chunk_fwd with separate workspaces.
 *  - The array holds GDN_CHUNK_MIN_WORKSPACE_BYTES, so dk = 128 always takes the fused
 *    single-kernel path. Returns GDN_ERR_WORKSPACE_TOO_SMALL if a path would need more
 *    workspace than the array holds (none does today).
 *  - A device-side timeout is recorded in the shared array: gdn_check_device_status(NULL,
 *    stream) reads it for the current device. */
gdn_status gdn_chunk_fwd_noalloc(const gdn_chunk_args* args, gdn_stream_t stream);

/* Bytes of device workspace for the fastest kda_chunk_fwd path with these arguments; 0 when
 * the arguments are invalid. For dk = 128 that is the status word plus the staging of the
 * two-kernel path: per 64-token chunk slot and v-head, W (transposed, as for
 * gdn_chunk_fwd_workspace_size), T diag(beta), the intra-chunk P = decay-weighted Q K^T, Q and
 * K scaled by their per-channel decays (all bf16 hi + lo) and the chunk's per-channel total
 * decay -- 113 KB (129 KB without W QDQ) for each of (B T / 64 + N) x Hv slots. Otherwise
 * GDN_CHUNK_MIN_WORKSPACE_BYTES. */
size_t kda_chunk_fwd_workspace_size(const gdn_chunk_args* args);

/* KDA variant ([K]): same contract with g [B, T, Hv, dk], one log-decay per key channel;
 * pairwise decays come from differences of prefix sums of g within a chunk. With
 * kda_chunk_fwd_workspace_size(args) bytes or more (and g 16-byte aligned), dk = 128 runs as
 * two tensor-core kernels (every chunk's state-independent work in parallel, then the state
 * carry); otherwise on CUDA cores, chunk by chunk (slower, same arithmetic). */
gdn_status kda_chunk_fwd(const gdn_chunk_args* args, void* workspace, size_t workspace_bytes,
                         gdn_stream_t stream);

/* Gradients of the forward with straight-through state QDQ ("Torch GDN/KDA decode QAT with INT8
 * recurrent state", "Megatron-Core QAT/QAD workflow" step 4: recurrent surrogate gradients,
 * identity straight-through estimator through QDQ; [F]: identity straight-through gradients).
 * For L = <o, dout> + <hT, dhT>, the derivatives of the token recurrence whose forward values
 * carry the state QDQ of GDN_FLAG_STATE_QDQ (either codec) and whose backward treats that QDQ as
 * the identity. All device fp32: dout [B, T, Hv, dv] (16-byte aligned); dhT [N, Hv, dk, dv] or NULL
 * (zero); outputs dq, dk [B, T, Hqk, dk] (summed over the value heads that share a q/k head),
 * dv [B, T, Hv, dv] (16-byte aligned), dg [B, T, Hv] (kda_chunk_bwd: [B, T, Hv, dk]),
 * dbeta [B, T, Hv], dh0 [N, Hv, dk, dv] or NULL. */
typedef struct {
  const float* dout;
  const float* dhT;
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dh0;
} gdn_chunk_grads;

/* Workspace of gdn_chunk_bwd (0 for invalid arguments): the status word, the state entering every
 * 64-token chunk (per chunk slot and v-head), per CTA (at most 152) the 16 sub-chunk checkpoints
 * of one 64-column state slab, and the per-slab, per-value-head dq, dk, dbeta, dg before their
 * sums (dbeta and the GDN dg also per dk / 32 key-row groups). */
size_t gdn_chunk_bwd_workspace_size(const gdn_chunk_args* args);
/* The backward on CUDA cores: per (sequence, head, 64-column value slab) a forward pass that
 * stores the chunk-entry states, then the chunks in reverse, each recomputed in 4-token sub-chunks
 * and walked token by token with the state gradient in registers; a second kernel sums the slab
 * (and, with GQA, value-head) partials of dq, dk, dbeta and dg in a fixed order. With
 * kda_chunk_bwd, g must be 16-byte aligned (else GDN_ERR_INVALID_ARG). args: the forward's inputs and flags (o, hT unused and may be NULL);
 * GDN_FLAG_W_QDQ and state_scales are refused (GDN_ERR_INVALID_ARG): the straight-through gradient
 * of the W QDQ belongs to the chunked form, which this backward does not take. */
gdn_status gdn_chunk_bwd(const gdn_chunk_args* args, const gdn_chunk_grads* grads, void* workspace,
                         size_t workspace_bytes, gdn_stream_t stream);
/* KDA (g [B, T, Hv, dk], dg [B, T, Hv, dk]). */
size_t kda_chunk_bwd_workspace_size(const gdn_chunk_args* args);
gdn_status kda_chunk_bwd(const gdn_chunk_args* args, const gdn_chunk_grads* grads, void* workspace,
                         size_t workspace_bytes, gdn_stream_t stream);

/* Prefill -> decode handoff ([H]: "Torch GDN/KDA decode QAT with INT8 recurrent state",
 * "Megatron-Core QAT/QAD workflow", steps 2-3 and the "Ordinary state-QDQ path" flowchart).
 * Per sequence n of length L_n, the first P_n = prefill_lengths_host[n] tokens run as chunked
 * prefill from h0 whose state is NOT quantized inside the prefix (W QDQ as GDN_FLAG_W_QDQ
 * asks); when P_n < L_n, the state is QDQ'd at the handoff (GDN_FLAG_STATE_QDQ) and every
 * remaining token is a decode step on the sequence's own q, k, v, g, beta (teacher forced):
 * read the state, decay, delta update, o from the updated state, then QDQ
 * (GDN_FLAG_STATE_QDQ) before the state is stored for the next token. o is written for every
 * token; hT (required, device fp32 [N, Hv, dk, dv], may alias h0 exactly) receives the final
 * state: the prefill state itself when P_n == L_n.
 * prefill_lengths_host: HOST int32 [N], 0 <= P_n <= L_n (else GDN_ERR_INVALID_ARG), read before
 * the call returns. Other arguments and layouts as gdn_chunk_fwd / kda_chunk_fwd. workspace:
 * device, 256-byte aligned, at least *_prefill_decode_workspace_size(args) bytes (else
 * GDN_ERR_WORKSPACE_TOO_SMALL): the prefill's staging plus a device copy of the prefill lengths.
 * Launches: the prefill kernels, then one CTA per (sequence, head) that keeps the state on chip
 * across all of the sequence's decode tokens. */
size_t gdn_prefill_decode_workspace_size(const gdn_chunk_args* args);
gdn_status gdn_prefill_decode_fwd(const gdn_chunk_args* args, const int32_t* prefill_lengths_host,
                                  void* workspace, size_t workspace_bytes, gdn_stream_t stream);
/* The same schedule for KDA (g [B, T, Hv, dk]). */
size_t kda_prefill_decode_workspace_size(const gdn_chunk_args* args);
gdn_status kda_prefill_decode_fwd(const gdn_chunk_args* args, const int32_t* prefill_lengths_host,
                                  void* workspace, size_t workspace_bytes, gdn_stream_t stream);

/* One decode token per sequence ([D], [R]). q, k: device bf16 [N, Hqk, dk]; v: device
 * bf16 [N, Hv, dv]; g: device fp32 [N, Hv] (GDN_FLAG_KDA: [N, Hv, dk]); beta: device fp32
 * [N, Hv]; state: device fp32 [N, Hv, dk, dv], read and overwritten in place; o: device
 * fp32 [N, Hv, dv]. Order per (sequence, head): read S, decay, delta update, o from the
 * updated state, then (GDN_FLAG_STATE_QDQ) per-tile E4M3 QDQ (GDN_FLAG_STATE_INT8: INT8 blocks),
 * then store S. */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state, float* o, int32_t N, int32_t Hqk,
                           int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                           gdn_stream_t stream);

/* Standalone dynamic tile QDQ ([F]: E4M3, scale amax / 448, 1 for an all-zero tile). x, y: device fp32
 * [lead, rows, cols] (y may equal x); a tile is all `rows` rows x `tile_cols` columns of one
 * leading index (the last tile may be narrower). scales: device fp32 [lead, ceil(cols /
 * tile_cols)] or NULL. Per tile, in fp32 with IEEE round-to-nearest: amax = max |x|,
 * s = amax / 448 (s == 0 -> 1), c = E4M3 round-to-nearest-even with saturation (x / s),
 * y = c * s. State tiles: rows = dk, tile_cols = 64. W tiles: rows = 64, tile_cols = dk. */
gdn_status fp8_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int32_t rows,
                        int32_t cols, int32_t tile_cols, gdn_stream_t stream);

/* Standalone INT8 block QDQ ([I]). x, y: device fp32 [rows, cols] (y may equal x); a block is
 * block_cols consecutive columns of one row (the last block of a row may be narrower). scales:
 * device fp32 [rows, ceil(cols / block_cols)] or NULL. Per block, in fp32 with IEEE
 * round-to-nearest: amax = max |x|, s = amax / 127 (s == 0 -> 1), c = the integer nearest x / s
 * (ties to even) within [-127, 127], y = c * s. The state codec: rows = N Hv dk (one per key row
 * of every state), cols = dv, block_cols = 32. */
gdn_status int8_block_qdq(const float* x, float* y, float* scales, int64_t rows, int32_t cols,
                          int32_t block_cols, gdn_stream_t stream);

/* Static description of a status code. */
const char* gdn_status_string(gdn_status status);

/* Synchronizes `stream`, then reads the status word a chunk-forward call left in
 * `workspace`: GDN_OK, or GDN_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait.
 * workspace == NULL reads the array behind gdn_chunk_fwd_noalloc on the current device. */
gdn_status gdn_check_device_status(const void* workspace, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNQAT_H */
