// gdn_verify_k128.cu -- verify and native-snapshot kernels for head width 128, scalar decay.
#include "gdn_verify_impl.cuh"

namespace gdn {

int launch_verify_k128(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                      cudaStream_t stream) {
  return dispatch_native<128, false>(p, qkv_dtype, state_dtype, native, stream);
}

}  // namespace gdn
