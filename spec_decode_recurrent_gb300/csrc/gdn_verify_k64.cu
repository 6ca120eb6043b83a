// gdn_verify_k64.cu -- verify and native-snapshot kernels for head width 64, both gate kinds.
#include "gdn_verify_impl.cuh"

namespace gdn {

int launch_verify_k64(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                     cudaStream_t stream) {
  return dispatch_native<64, false>(p, qkv_dtype, state_dtype, native, stream);
}

int launch_verify_k64_kda(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                         cudaStream_t stream) {
  return dispatch_native<64, true>(p, qkv_dtype, state_dtype, native, stream);
}

}  // namespace gdn
