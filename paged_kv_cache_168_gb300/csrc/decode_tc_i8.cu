// decode_tc_i8.cu -- launcher of the tensor-core decode kernel for 8-bit caches
// (the kernel itself is in decode_tc.cuh).
#include "decode_tc.cuh"

namespace pkv {

cudaError_t launch_decode_tc_i8(const DecodeParams& p, int act_dtype, int group, int num_sms, cudaStream_t stream) {
  if (p.num_seqs > kTcI8MaxSeqs || group < 1 || group > 8) return cudaErrorInvalidValue;
  cudaError_t e;
  if (act_dtype == PA_F16)
    e = launch_group<__half, kI8Stages, true, kI8Raw>(p, group, num_sms, stream);
  else if (act_dtype == PA_BF16)
    e = launch_group<__nv_bfloat16, kI8Stages, true, kI8Raw>(p, group, num_sms, stream);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_merge(p, act_dtype, kD, stream);
}

}  // namespace pkv
