// gdnqat_api.cu -- the extern "C" surface declared in include/gdnqat.h.
//
// Every entry point validates its arguments on the host, then probes the current device,
// and only then enqueues work; a non-OK status means nothing was launched (per "GDN state/W QAT
// foundation", unmet hardware or version requirements fail with an error before any kernel
// runs). The library allocates nothing.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace {

using gdn::ChunkProblem;

constexpr int kMaxDevices = 64;
std::atomic<int> g_arch_ok[kMaxDevices];   // 0 = unknown, 1 = sm_103, 2 = other (devices >= 64 are probed every call)

}  // namespace

namespace gdn {
gdn_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return GDN_ERR_UNSUPPORTED_ARCH;
  }
  if (dev < kMaxDevices) {
    const int known = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (known) return known == 1 ? GDN_OK : GDN_ERR_UNSUPPORTED_ARCH;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return GDN_ERR_UNSUPPORTED_ARCH;
  }
  const bool ok = (major == 10 && minor == 3);
  if (dev < kMaxDevices) g_arch_ok[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? GDN_OK : GDN_ERR_UNSUPPORTED_ARCH;
}
}  // namespace gdn

namespace {
using gdn::check_device;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool dk_ok(int dk) { return dk == 64 || dk == 128; }

// the kernels' state-QDQ selector: 0 off, 1 E4M3 tiles, 2 INT8 blocks
int state_codec(uint32_t flags) {
  if (!(flags & GDN_FLAG_STATE_QDQ)) return 0;
  return (flags & GDN_FLAG_STATE_INT8) ? 2 : 1;
}
bool dv_ok(int dv) { return dv == 64 || dv == 128 || dv == 256; }

constexpr size_t kWorkspaceBytes = gdn::kStatusBytes;   // device status word (+ padding to one line)
static_assert(kWorkspaceBytes == GDN_CHUNK_MIN_WORKSPACE_BYTES, "the header's minimum must match");

gdn_status validate_chunk(const gdn_chunk_args* a, bool kda, bool need_o = true) {
  if (!a) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->T < 0 || a->N < 0 || a->Hqk <= 0 || a->Hv <= 0 || a->dk <= 0 || a->dv <= 0)
    return GDN_ERR_INVALID_ARG;
  if (a->Hv % a->Hqk != 0) return GDN_ERR_INVALID_ARG;
  if (a->flags & ~(GDN_FLAG_STATE_QDQ | GDN_FLAG_W_QDQ | GDN_FLAG_STATE_INT8)) return GDN_ERR_INVALID_ARG;
  if (!dk_ok(a->dk) || !dv_ok(a->dv)) return GDN_ERR_UNSUPPORTED_SHAPE;
  const int64_t tokens = (int64_t)a->B * a->T;
  if (a->cu_seqlens) {
    if (a->B != 1 || a->N < 1 || !a->cu_seqlens_host) return GDN_ERR_INVALID_ARG;
    const int32_t* c = a->cu_seqlens_host;
    if (c[0] != 0 || c[a->N] != a->T) return GDN_ERR_INVALID_ARG;
    for (int n = 0; n < a->N; ++n)
      if (c[n + 1] < c[n]) return GDN_ERR_INVALID_ARG;
  } else if (a->N != a->B) {
    return GDN_ERR_INVALID_ARG;
  }
  if (tokens > 0) {
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || (need_o && !a->o)) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) ||
        !aligned(a->g, 4) || !aligned(a->beta, 4))
      return GDN_ERR_INVALID_ARG;
  }
  if ((a->h0 && !aligned(a->h0, 16)) || (a->hT && !aligned(a->hT, 16))) return GDN_ERR_INVALID_ARG;
  const size_t st = (size_t)a->N * a->Hv * a->dk * a->dv * 4;
  const size_t nq = (size_t)tokens * a->Hqk * a->dk * 2, nv = (size_t)tokens * a->Hv * a->dv * 2;
  const size_t ng = (size_t)tokens * a->Hv * 4 * (kda ? a->dk : 1), nb = (size_t)tokens * a->Hv * 4;
  const size_t no = (size_t)tokens * a->Hv * a->dv * 4;
  // o must not alias any input; hT may alias h0 only exactly
  if (overlaps(a->o, no, a->q, nq) || overlaps(a->o, no, a->k, nq) || overlaps(a->o, no, a->v, nv) ||
      overlaps(a->o, no, a->g, ng) || overlaps(a->o, no, a->beta, nb) || overlaps(a->o, no, a->h0, st) ||
      overlaps(a->o, no, a->hT, st))
    return GDN_ERR_INVALID_ARG;
  if (a->hT && a->h0 && a->hT != a->h0 && overlaps(a->hT, st, a->h0, st)) return GDN_ERR_INVALID_ARG;
  if (a->state_scales) {   // final-state QDQ scales: only with the state quantizer on
    if (!(a->flags & GDN_FLAG_STATE_QDQ) || !aligned(a->state_scales, 4)) return GDN_ERR_INVALID_ARG;
    const size_t ns = (a->flags & GDN_FLAG_STATE_INT8)
                          ? (size_t)a->N * a->Hv * a->dk * ((a->dv + 31) / 32) * 4
                          : (size_t)a->N * a->Hv * ((a->dv + 63) / 64) * 4;
    if (overlaps(a->state_scales, ns, a->o, no) || overlaps(a->state_scales, ns, a->hT, st) ||
        overlaps(a->state_scales, ns, a->h0, st))
      return GDN_ERR_INVALID_ARG;
  }
  return GDN_OK;
}

gdn_status chunk_fwd(const gdn_chunk_args* a, void* ws, size_t ws_bytes, cudaStream_t stream, bool kda) {
  gdn_status s = validate_chunk(a, kda);
  if (s != GDN_OK) return s;
  if (!ws || ws_bytes < kWorkspaceBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return GDN_ERR_INVALID_ARG;
  s = check_device();
  if (s != GDN_OK) return s;
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return GDN_ERR_CUDA;
  if ((int64_t)a->N * a->Hv == 0) return GDN_OK;
  ChunkProblem p{a->q, a->k, a->v, a->g, a->beta, a->h0, a->cu_seqlens, a->o, a->hT,
                 a->B, a->T, a->N, a->Hqk, a->Hv, a->dk, a->dv, a->scale,
                 state_codec(a->flags), (a->flags & GDN_FLAG_W_QDQ) ? 1 : 0, kda ? 1 : 0};
  p.cu_host = a->cu_seqlens ? a->cu_seqlens_host : nullptr;
  p.state_scales = a->state_scales;
  // dk = 128: the two-kernel path (parallel prep, then the state chain) when the workspace
  // holds its staging, else (GDN) the single fused kernel; other shapes and KDA with a small
  // workspace: CUDA cores
  cudaError_t e;
  if (gdn::kda_split_supported(p) && ws_bytes >= gdn::kda_split_layout(p).total)
    e = gdn::launch_kda_split(p, ws, stream);
  else if (gdn::chunk_split_supported(p) && ws_bytes >= gdn::chunk_split_layout(p).total)
    e = gdn::launch_chunk_split(p, ws, stream);
  else if (gdn::chunk_tc_supported(p))
    e = gdn::launch_chunk_tc(p, static_cast<int*>(ws), stream);
  else
    e = gdn::launch_chunk_simt(p, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The prefill part of a prefill -> decode handoff runs the two-kernel tensor-core paths (or CUDA
// cores for the shapes they do not take); the device copy of the prefill lengths follows the
// chunk workspace.
size_t handoff_chunk_bytes(const ChunkProblem& p) {
  if (gdn::kda_split_supported(p)) return gdn::kda_split_layout(p).total;
  if (gdn::chunk_split_supported(p)) return gdn::chunk_split_layout(p).total;
  return kWorkspaceBytes;
}
size_t handoff_lens_offset(const ChunkProblem& p) { return (handoff_chunk_bytes(p) + 255) & ~(size_t)255; }
size_t handoff_bytes(const ChunkProblem& p) { return handoff_lens_offset(p) + (size_t)p.N * 4; }

ChunkProblem problem_of(const gdn_chunk_args* a, bool kda) {
  ChunkProblem p{a->q, a->k, a->v, a->g, a->beta, a->h0, a->cu_seqlens, a->o, a->hT,
                 a->B, a->T, a->N, a->Hqk, a->Hv, a->dk, a->dv, a->scale,
                 state_codec(a->flags), (a->flags & GDN_FLAG_W_QDQ) ? 1 : 0, kda ? 1 : 0};
  p.cu_host = a->cu_seqlens ? a->cu_seqlens_host : nullptr;
  p.state_scales = a->state_scales;
  return p;
}

gdn_status prefill_decode(const gdn_chunk_args* a, const int32_t* plens, void* ws, size_t ws_bytes,
                          cudaStream_t stream, bool kda) {
  gdn_status s = validate_chunk(a, kda);
  if (s != GDN_OK) return s;
  if (!a->hT) return GDN_ERR_INVALID_ARG;   // the handed-off state lives in hT
  if (a->N > 0 && !plens) return GDN_ERR_INVALID_ARG;
  for (int n = 0; n < a->N; ++n) {
    const int64_t L = a->cu_seqlens ? (int64_t)a->cu_seqlens_host[n + 1] - a->cu_seqlens_host[n] : (int64_t)a->T;
    if (plens[n] < 0 || plens[n] > L) return GDN_ERR_INVALID_ARG;
  }
  ChunkProblem p = problem_of(a, kda);
  if (!ws || ws_bytes < handoff_bytes(p)) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return GDN_ERR_INVALID_ARG;
  s = check_device();
  if (s != GDN_OK) return s;
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return GDN_ERR_CUDA;
  if ((int64_t)a->N * a->Hv == 0) return GDN_OK;
  int32_t* lens = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) + handoff_lens_offset(p));
  // pageable source: the copy is staged before the call returns
  if (cudaMemcpyAsync(lens, plens, (size_t)p.N * 4, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  // the prefix: chunked, W QDQ as asked, no state QDQ
  const int state_qdq = p.state_qdq;
  float* const state_scales = p.state_scales;
  p.state_qdq = 0;
  p.state_scales = nullptr;   // the prefix leaves its state unquantized; the decode part writes the scales
  p.lens = lens;
  p.lens_host = plens;
  cudaError_t e;
  if (gdn::kda_split_supported(p))
    e = gdn::launch_kda_split(p, ws, stream);
  else if (gdn::chunk_split_supported(p))
    e = gdn::launch_chunk_split(p, ws, stream);
  else
    e = gdn::launch_chunk_simt(p, stream);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  // the handoff and the decode tokens
  p.state_qdq = state_qdq;
  p.state_scales = state_scales;
  return gdn::launch_handoff_suffix(p, lens, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// ---- backward ----
bool bwd_shape_ok(const gdn_chunk_args* a) { return !(a->flags & GDN_FLAG_W_QDQ); }

gdn_status chunk_bwd(const gdn_chunk_args* a, const gdn_chunk_grads* gr, void* ws, size_t ws_bytes,
                     cudaStream_t stream, bool kda) {
  gdn_status s = validate_chunk(a, kda, false);
  if (s != GDN_OK) return s;
  // the straight-through gradient of W QDQ lives in the chunked form, which this backward does not take
  if (!bwd_shape_ok(a) || a->state_scales) return GDN_ERR_INVALID_ARG;
  if (!gr) return GDN_ERR_INVALID_ARG;
  const int64_t tokens = (int64_t)a->B * a->T;
  if (tokens > 0) {
    if (!gr->dout || !gr->dq || !gr->dk || !gr->dv || !gr->dg || !gr->dbeta) return GDN_ERR_INVALID_ARG;
    if (!aligned(gr->dout, 16) || !aligned(gr->dv, 16) || !aligned(gr->dq, 4) || !aligned(gr->dk, 4) ||
        !aligned(gr->dg, 4) || !aligned(gr->dbeta, 4))
      return GDN_ERR_INVALID_ARG;
    if (kda && !aligned(a->g, 16)) return GDN_ERR_INVALID_ARG;   // staged in 16-byte copies
  }
  if ((gr->dhT && !aligned(gr->dhT, 16)) || (gr->dh0 && !aligned(gr->dh0, 16))) return GDN_ERR_INVALID_ARG;
  ChunkProblem p = problem_of(a, kda);
  p.state_scales = nullptr;
  if (!ws || ws_bytes < gdn::chunk_bwd_layout(p).total) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return GDN_ERR_INVALID_ARG;
  s = check_device();
  if (s != GDN_OK) return s;
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return GDN_ERR_CUDA;
  const gdn::BwdGrads g{gr->dout, gr->dhT, gr->dq, gr->dk, gr->dv, gr->dg, gr->dbeta, gr->dh0};
  return gdn::launch_chunk_bwd(p, g, ws, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t bwd_workspace(const gdn_chunk_args* a, bool kda) {
  if (validate_chunk(a, kda, false) != GDN_OK || !bwd_shape_ok(a)) return 0;
  return gdn::chunk_bwd_layout(problem_of(a, kda)).total;
}

}  // namespace

extern "C" {

size_t gdn_chunk_bwd_workspace_size(const gdn_chunk_args* args) { return bwd_workspace(args, false); }
size_t kda_chunk_bwd_workspace_size(const gdn_chunk_args* args) { return bwd_workspace(args, true); }

gdn_status gdn_chunk_bwd(const gdn_chunk_args* args, const gdn_chunk_grads* grads, void* workspace,
                         size_t workspace_bytes, gdn_stream_t stream) {
  return chunk_bwd(args, grads, workspace, workspace_bytes, (cudaStream_t)stream, false);
}

gdn_status kda_chunk_bwd(const gdn_chunk_args* args, const gdn_chunk_grads* grads, void* workspace,
                         size_t workspace_bytes, gdn_stream_t stream) {
  return chunk_bwd(args, grads, workspace, workspace_bytes, (cudaStream_t)stream, true);
}

size_t gdn_prefill_decode_workspace_size(const gdn_chunk_args* args) {
  if (validate_chunk(args, false) != GDN_OK) return 0;
  return handoff_bytes(problem_of(args, false));
}

size_t kda_prefill_decode_workspace_size(const gdn_chunk_args* args) {
  if (validate_chunk(args, true) != GDN_OK) return 0;
  return handoff_bytes(problem_of(args, true));
}

gdn_status gdn_prefill_decode_fwd(const gdn_chunk_args* args, const int32_t* prefill_lengths_host, void* workspace,
                                  size_t workspace_bytes, gdn_stream_t stream) {
  return prefill_decode(args, prefill_lengths_host, workspace, workspace_bytes, (cudaStream_t)stream, false);
}

gdn_status kda_prefill_decode_fwd(const gdn_chunk_args* args, const int32_t* prefill_lengths_host, void* workspace,
                                  size_t workspace_bytes, gdn_stream_t stream) {
  return prefill_decode(args, prefill_lengths_host, workspace, workspace_bytes, (cudaStream_t)stream, true);
}

const char* gdn_status_string(gdn_status status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED_ARCH: return "unsupported device (needs sm_103 / GB300)";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (dk in {64,128}, dv in {64,128,256})";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_CUDA: return "CUDA error";
    case GDN_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
  }
  return "unknown status";
}

size_t gdn_chunk_fwd_workspace_size(const gdn_chunk_args* args) {
  const bool gdn_ok = validate_chunk(args, false) == GDN_OK;
  if (!gdn_ok && validate_chunk(args, true) != GDN_OK) return 0;
  if (gdn_ok) {
    const gdn::ChunkProblem p{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                              args->B, args->T, args->N, args->Hqk, args->Hv, args->dk, args->dv, args->scale,
                              state_codec(args->flags), (args->flags & GDN_FLAG_W_QDQ) ? 1 : 0, 0};
    if (gdn::chunk_split_supported(p)) return gdn::chunk_split_layout(p).total;
  }
  return kWorkspaceBytes;
}

size_t kda_chunk_fwd_workspace_size(const gdn_chunk_args* args) {
  if (validate_chunk(args, true) != GDN_OK) return 0;
  const gdn::ChunkProblem p{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                            args->B, args->T, args->N, args->Hqk, args->Hv, args->dk, args->dv, args->scale,
                            state_codec(args->flags), (args->flags & GDN_FLAG_W_QDQ) ? 1 : 0, 1};
  if (gdn::kda_split_supported(p)) return gdn::kda_split_layout(p).total;
  return kWorkspaceBytes;
}

gdn_status gdn_chunk_fwd(const gdn_chunk_args* args, void* workspace, size_t workspace_bytes,
                         gdn_stream_t stream) {
  return chunk_fwd(args, workspace, workspace_bytes, (cudaStream_t)stream, false);
}

gdn_status kda_chunk_fwd(const gdn_chunk_args* args, void* workspace, size_t workspace_bytes,
                         gdn_stream_t stream) {
  return chunk_fwd(args, workspace, workspace_bytes, (cudaStream_t)stream, true);
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                           float* state, float* o, int32_t N, int32_t Hqk, int32_t Hv, int32_t dk, int32_t dv,
                           float scale, uint32_t flags, gdn_stream_t stream) {
  if (N < 0 || Hqk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hqk != 0) return GDN_ERR_INVALID_ARG;
  if (flags & ~(GDN_FLAG_STATE_QDQ | GDN_FLAG_KDA | GDN_FLAG_STATE_INT8)) return GDN_ERR_INVALID_ARG;
  if (!dk_ok(dk) || !dv_ok(dv)) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (N > 0) {
    if (!q || !k || !v || !g || !beta || !state || !o) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state, 16) || !aligned(o, 16) ||
        !aligned(g, 4) || !aligned(beta, 4))
      return GDN_ERR_INVALID_ARG;
    const size_t st = (size_t)N * Hv * dk * dv * 4, no = (size_t)N * Hv * dv * 4;
    if (overlaps(o, no, state, st) || overlaps(o, no, q, (size_t)N * Hqk * dk * 2) ||
        overlaps(o, no, k, (size_t)N * Hqk * dk * 2) || overlaps(o, no, v, (size_t)N * Hv * dv * 2))
      return GDN_ERR_INVALID_ARG;
  }
  gdn_status s = check_device();
  if (s != GDN_OK) return s;
  return gdn::launch_decode(q, k, v, g, beta, state, o, N, Hqk, Hv, dk, dv, scale,
                            state_codec(flags), (flags & GDN_FLAG_KDA) ? 1 : 0,
                            (cudaStream_t)stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status fp8_tile_qdq(const float* x, float* y, float* scales, int64_t lead, int32_t rows, int32_t cols,
                        int32_t tile_cols, gdn_stream_t stream) {
  if (lead < 0 || rows < 0 || cols < 0 || tile_cols <= 0) return GDN_ERR_INVALID_ARG;
  const size_t n = (size_t)lead * rows * cols * 4;
  if (n > 0 && (!x || !y || !aligned(x, 4) || !aligned(y, 4))) return GDN_ERR_INVALID_ARG;
  if (x != y && overlaps(x, n, y, n)) return GDN_ERR_INVALID_ARG;
  if (scales && !aligned(scales, 4)) return GDN_ERR_INVALID_ARG;
  gdn_status s = check_device();
  if (s != GDN_OK) return s;
  return gdn::launch_tile_qdq(x, y, scales, lead, rows, cols, tile_cols, (cudaStream_t)stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status int8_block_qdq(const float* x, float* y, float* scales, int64_t rows, int32_t cols, int32_t block_cols,
                          gdn_stream_t stream) {
  if (rows < 0 || cols < 0 || block_cols <= 0) return GDN_ERR_INVALID_ARG;
  const size_t n = (size_t)rows * cols * 4;
  if (n > 0 && (!x || !y || !aligned(x, 4) || !aligned(y, 4))) return GDN_ERR_INVALID_ARG;
  if (x != y && overlaps(x, n, y, n)) return GDN_ERR_INVALID_ARG;
  if (scales && !aligned(scales, 4)) return GDN_ERR_INVALID_ARG;
  gdn_status s = check_device();
  if (s != GDN_OK) return s;
  return gdn::launch_int8_block_qdq(x, y, scales, rows, cols, block_cols, (cudaStream_t)stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status gdn_check_device_status(const void* workspace, gdn_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  int word = 0;
  if (!workspace) {   // the array behind gdn_chunk_fwd_noalloc on the current device
    const gdn_status s = gdn::noalloc_status_word(&word);
    if (s != GDN_OK) return s;
  } else if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    return GDN_ERR_CUDA;
  }
  return word == 0 ? GDN_OK : GDN_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
