// quotient_sweep.cu -- the standalone QDQ ops' quotient (gdn::quotient / gdn::quotient2 of
// common.cuh: the reciprocal of the scale plus two FMA corrections) against the IEEE divide,
// over every significand of one operand.
//
// mode 0: x runs over all 2^23 significands of [1, 2), scaled by 2^exps[e] for each listed
//         exponent; s runs over the list `vals`.
// mode 1: s runs over all 2^23 significands of [1, 2), scaled by 2^exps[e]; x over `vals`.
// Per pair: the quotient bits against __fdiv_rn (counts[0]), the E4M3 codes (round to nearest
// even, satfinite) of both (counts[1]), the paired form against the scalar form (counts[2]), and
// for reference the codes of x times the rounded reciprocal alone, the fused kernels' QDQ
// (counts[3]). The first mismatching pair of counts[0] or counts[1] lands in first[0..1].
#include "../../fp8_state_qat_gb300/csrc/common.cuh"

namespace {

__device__ __forceinline__ unsigned char e4m3(float y) {
  return (unsigned char)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
}

__global__ void sweep_kernel(const float* vals, int nvals, const int* exps, int nexps, int mode,
                             unsigned long long* counts, unsigned int* first) {
  const unsigned long long total = (1ull << 23) * (unsigned long long)nvals * (unsigned long long)nexps;
  unsigned long long local[4] = {0, 0, 0, 0};
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < total;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const unsigned int m = (unsigned int)(i & ((1u << 23) - 1));
    const unsigned long long rest = i >> 23;
    const int vi = (int)(rest % (unsigned long long)nvals), ei = (int)(rest / (unsigned long long)nvals);
    const float swept = __uint_as_float(((unsigned int)(127 + exps[ei]) << 23) | m);
    const float x = mode == 0 ? swept : vals[vi];
    const float s = mode == 0 ? vals[vi] : swept;
    const float r = __frcp_rn(s);
    const float q = gdn::quotient(x, s, r);
    const float2 q2 = gdn::quotient2(make_float2(x, -x), make_float2(-s, -s), make_float2(r, r));
    const float qr = __fdiv_rn(x, s);
    const bool bad_bits = __float_as_uint(q) != __float_as_uint(qr);
    const bool bad_code = e4m3(q) != e4m3(qr);
    local[0] += bad_bits;
    local[1] += bad_code;
    local[2] += (__float_as_uint(q2.x) != __float_as_uint(q)) || (__float_as_uint(q2.y) != __float_as_uint(-q));
    local[3] += e4m3(__fmul_rn(x, r)) != e4m3(qr);
    if ((bad_bits || bad_code) && atomicCAS(first + 2, 0u, 1u) == 0u) {
      first[0] = __float_as_uint(x);
      first[1] = __float_as_uint(s);
    }
  }
  for (int k = 0; k < 4; ++k)
    if (local[k]) atomicAdd(counts + k, local[k]);
}

}  // namespace

// vals: device fp32 [nvals]; exps: device int32 [nexps] (each in [-100, 100]); counts: device
// uint64 [4], zeroed by the caller; first: device uint32 [3], zeroed by the caller.
extern "C" int gdnqat_testing_quotient_sweep(const float* vals, int nvals, const int* exps, int nexps, int mode,
                                             unsigned long long* counts, unsigned int* first, cudaStream_t stream) {
  if (nvals <= 0 || nexps <= 0 || (mode != 0 && mode != 1)) return 1;
  sweep_kernel<<<152 * 8, 256, 0, stream>>>(vals, nvals, exps, nexps, mode, counts, first);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

namespace {
// gdn::qdq_scale(amax) against the IEEE divide with the zero guard, for every non-negative finite
// fp32 amax (bit patterns 0 .. 0x7f7fffff): mismatches counted in counts[0], the first in first[0].
__global__ void scale_sweep_kernel(unsigned long long* counts, unsigned int* first) {
  unsigned long long local = 0;
  for (unsigned int b = blockIdx.x * blockDim.x + threadIdx.x; b <= 0x7f7fffffu; b += gridDim.x * blockDim.x) {
    const float x = __uint_as_float(b);
    float want = __fdiv_rn(x, 448.0f);
    if (want == 0.0f) want = 1.0f;
    if (__float_as_uint(gdn::qdq_scale(x)) != __float_as_uint(want)) {
      ++local;
      atomicCAS(first, 0u, b);
    }
    if (b > 0x7f7fffffu - gridDim.x * blockDim.x) break;   // the next step would wrap around
  }
  if (local) atomicAdd(counts, local);
}
}  // namespace

extern "C" int gdnqat_testing_scale_sweep(unsigned long long* counts, unsigned int* first, cudaStream_t stream) {
  scale_sweep_kernel<<<152 * 8, 256, 0, stream>>>(counts, first);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
