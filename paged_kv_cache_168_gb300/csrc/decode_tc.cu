// decode_tc.cu -- launcher of the tensor-core decode kernel for 16-bit caches
// (the kernel itself is in decode_tc.cuh).
#include "decode_tc.cuh"

namespace pkv {

cudaError_t launch_decode_tc(const DecodeParams& p, int dtype, int group, int num_sms, cudaStream_t stream) {
  if (p.num_seqs > kTcMaxSeqs) return cudaErrorInvalidValue;
  const bool three = p.num_seqs <= 512;    // shared memory: 3 stages + item ordering of <= 512 sequences
  cudaError_t e;
  if (dtype == PA_F16)
    e = three ? launch_group<__half, 3, false, 1>(p, group, num_sms, stream)
              : launch_group<__half, 2, false, 1>(p, group, num_sms, stream);
  else if (dtype == PA_BF16)
    e = three ? launch_group<__nv_bfloat16, 3, false, 1>(p, group, num_sms, stream)
              : launch_group<__nv_bfloat16, 2, false, 1>(p, group, num_sms, stream);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_merge(p, dtype, kD, stream);
}

}  // namespace pkv
