// decode_tc_prefix.cu -- launcher of the tensor-core decode kernel with shared
// prefixes (the kernel itself is in decode_tc.cuh): each group's prefix blocks
// are streamed once and serve every member sequence of the group.
#include "decode_tc.cuh"

namespace pkv {

namespace {
template <typename T>
cudaError_t launch_sp_group(const DecodeParams& p, int group, int num_sms, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_typed<T, 1, 3, false, 1, true>(p, num_sms, stream);
    case 2: return launch_typed<T, 2, 3, false, 1, true>(p, num_sms, stream);
    case 4: return launch_typed<T, 4, 3, false, 1, true>(p, num_sms, stream);
    case 8: return launch_typed<T, 8, 3, false, 1, true>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_decode_tc_sp(const DecodeParams& p, int dtype, int group, int num_sms, cudaStream_t stream) {
  if (p.num_seqs > kTcSpMaxSeqs || p.window > 0 || p.ring_blocks > 0) return cudaErrorInvalidValue;
  cudaError_t e;
  if (dtype == PA_F16) e = launch_sp_group<__half>(p, group, num_sms, stream);
  else if (dtype == PA_BF16) e = launch_sp_group<__nv_bfloat16>(p, group, num_sms, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_merge_sp(p, dtype, kD, stream);
}

}  // namespace pkv
