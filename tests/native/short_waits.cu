// short_waits.cu -- test-only entry to the two-kernel chunk forward built with GDN_WAIT_LIMIT=0
// (every pipeline wait of chunk_prep.cu / chunk_chain.cu gives up on its first poll).
//
// The kernels then take their abort path: the CTA raises its abort flag, both warpgroups leave
// their loops at their next checked barrier without issuing further MMAs or copies, the status
// word in the workspace is set, the TMA loads already in flight are waited for with their own
// (unchanged) limits and TMEM is freed. gdn_check_device_status on the same workspace must then
// report GDN_ERR_DEVICE_TIMEOUT, and the device must stay usable.
#include "../../fp8_state_qat_gb300/csrc/kernels.h"

extern "C" int gdnqat_testing_split_fwd(const gdn_chunk_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a || !ws || a->dk != 128 || a->dv % 64 != 0 || a->cu_seqlens || a->B != a->N) return 1;
  gdn::ChunkProblem p{a->q, a->k, a->v, a->g, a->beta, a->h0, nullptr, a->o, a->hT,
                      a->B, a->T, a->N, a->Hqk, a->Hv, a->dk, a->dv, a->scale,
                      (a->flags & GDN_FLAG_STATE_QDQ) ? 1 : 0, (a->flags & GDN_FLAG_W_QDQ) ? 1 : 0, 0};
  if (ws_bytes < gdn::chunk_split_layout(p).total) return 2;
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return 3;
  return gdn::launch_chunk_split(p, ws, stream) == cudaSuccess ? 0 : 4;
}
