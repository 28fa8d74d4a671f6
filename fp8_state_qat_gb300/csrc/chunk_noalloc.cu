// chunk_noalloc.cu -- gdn_chunk_fwd for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine at the point where they run
// the forward: code running inside a memory allocator's own hooks, latency-critical paths
// where an allocation's implicit device synchronization is not allowed, or processes whose
// device memory is fully handed out to a framework's pool. gdn_chunk_fwd needs at least a
// small device workspace (the status word of the tensor-core kernels' bounded waits); this
// variant takes that minimum from a fixed-size array that lives in the library itself, so
// the caller passes only its inputs and outputs (and the forward runs its single-kernel path).
//
// The array is a file-scope __device__ object: every GPU that loads the library holds these
// kNoAllocScratchBytes until the process exits, and all calls on a device share it. The host
// symbol is only a stand-in: each call looks up the array's device address on the current
// device with cudaGetSymbolAddress (cheap once the library's device code is loaded there; a
// looked-up address is never reused across calls, so a context that was reset and re-created
// cannot leave a stale one behind).
#include "../../include/gdnqat.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 256;   // the chunk forward's minimum workspace
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.
gdn_status scratch_for_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  *out = p;
  return GDN_OK;
}

}  // namespace

namespace gdn {
gdn_status noalloc_status_word(int* word) {
  gdn_status s = check_device();
  if (s != GDN_OK) return s;
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != GDN_OK) return s;
  return cudaMemcpy(word, scratch, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace gdn

extern "C" gdn_status gdn_chunk_fwd_noalloc(const gdn_chunk_args* args, gdn_stream_t stream) {
  if (gdn_chunk_fwd_workspace_size(args) == 0) {
    // invalid arguments: let the regular entry point report which check failed
    return gdn_chunk_fwd(args, nullptr, 0, stream);
  }
  // the smallest workspace gdn_chunk_fwd accepts (it then takes its single-kernel path)
  if (GDN_CHUNK_MIN_WORKSPACE_BYTES > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE_TOO_SMALL;
  // the device check comes first: on another GPU the array has no device image to look up
  gdn_status s = gdn::check_device();
  if (s != GDN_OK) return s;
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != GDN_OK) return s;
  // gdn_chunk_fwd clears the status word on `stream` before its kernel runs
  return gdn_chunk_fwd(args, scratch, kNoAllocScratchBytes, stream);
}
